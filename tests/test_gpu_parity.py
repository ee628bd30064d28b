"""GPU parity: every kernel against the fp64 oracle on the same seeded inputs.

Index scores and top-k index sets must match bit for bit (dyadic indexer
inputs make every fp32 sum exact). Attention outputs, LSE and gradients must
satisfy max|err| <= 2e-2 * max|ref| per tensor.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TOL, bf16_dev, dev, host_f64, rel_err

pytestmark = pytest.mark.gpu


def _dsa():
    import sparse_attention_index_gb300 as dsa
    return dsa


def _indexer_case(B, S, Hi, Di, seed, ndocs=0, w_kind="dyadic"):
    q = synth.dyadic_bf16((B, S, Hi, Di), seed, synth.STREAM_Q_IDX, -8, 8, 3)
    k = synth.dyadic_bf16((B, S, Di), seed, synth.STREAM_K_IDX, -8, 8, 3)
    if w_kind == "dyadic":
        w = synth.dyadic_f32((B, S, Hi), seed, synth.STREAM_W, -1, 1, 4)
    else:
        w = synth.signed_nonzero_f32((B, S, Hi), seed, synth.STREAM_W, 8, 3)
    seg = synth.segments(B, S, ndocs, seed) if ndocs else None
    return {"q_idx": q, "k_idx": k, "w": w, "seg": seg}


def _check_scores(gpu_scores, ref, rows, S):
    """Exact equality on s <= t (values; -0 == +0), -inf in the same places."""
    for r, row in enumerate(rows):
        b, t = divmod(int(row), S)
        g = gpu_scores[b, t, : t + 1]
        o = ref[r, : t + 1]
        assert np.array_equal(np.isneginf(g), np.isneginf(o)), (b, t)
        fin = np.isfinite(o)
        bad = np.nonzero(g[fin] != o[fin])[0]
        assert bad.size == 0, (b, t, bad[:5], g[fin][bad[:5]], o[fin][bad[:5]])


def _run_scores(inp, w_bf16=False):
    dsa = _dsa()
    w = dev(inp["w"])
    if w_bf16:
        w = w.to(torch.bfloat16)
    seg = None if inp["seg"] is None else dev(inp["seg"])
    sc = dsa.dsa_index_scores(bf16_dev(inp["q_idx"]), bf16_dev(inp["k_idx"]), w, seg)
    assert dsa.dsa_get_last_device_error() == 0
    return sc


# ------------------------------------------------------------------ indexer

INDEXER_CASES = [
    # B, S, Hi, Di, ndocs, w_kind
    (1, 128, 4, 32, 0, "signed_nonzero"),
    (2, 700, 64, 128, 0, "dyadic"),
    (1, 489, 64, 128, 3, "dyadic"),
    (1, 300, 1, 64, 0, "dyadic"),
    (1, 300, 8, 64, 2, "dyadic"),
    (1, 333, 16, 64, 0, "dyadic"),
    (1, 257, 32, 32, 0, "dyadic"),
    (2, 190, 128, 128, 0, "dyadic"),
]


@pytest.mark.parametrize("case", INDEXER_CASES)
def test_index_scores_exact(case):
    B, S, Hi, Di, ndocs, w_kind = case
    inp = _indexer_case(B, S, Hi, Di, seed=100 + S, ndocs=ndocs, w_kind=w_kind)
    sc = host_f64(_run_scores(inp))
    ref = oracle.index_scores(inp["q_idx"], inp["k_idx"], inp["w"], inp["seg"])
    _check_scores(sc, ref, np.arange(B * S), S)


def test_index_scores_bf16_weights():
    inp = _indexer_case(1, 260, 64, 128, seed=7)
    sc = host_f64(_run_scores(inp, w_bf16=True))
    ref = oracle.index_scores(inp["q_idx"], inp["k_idx"], inp["w"], None)
    _check_scores(sc, ref, np.arange(260), 260)


def test_index_scores_leading_dimension():
    dsa = _dsa()
    inp = _indexer_case(1, 150, 64, 128, seed=8)
    scores = torch.full((1, 150, 160), 7.0, device="cuda")
    dsa.dsa_index_scores(bf16_dev(inp["q_idx"]), bf16_dev(inp["k_idx"]), dev(inp["w"]), None,
                         scores=scores)
    ref = oracle.index_scores(inp["q_idx"], inp["k_idx"], inp["w"], None)
    _check_scores(host_f64(scores), ref, np.arange(150), 150)
    assert torch.all(scores[..., 150:] == 7.0)   # padding columns untouched


# ------------------------------------------------------------ fp8 indexer

FP8_CASES = [
    # B, S, Hi, Di, ndocs, k_scale
    (1, 128, 4, 32, 0, "none"),
    (2, 700, 64, 128, 0, "pow2"),
    (1, 489, 64, 128, 3, "pow2"),
    (1, 300, 1, 64, 0, "none"),
    (1, 300, 8, 64, 2, "pow2"),
    (1, 333, 16, 64, 0, "none"),
    (1, 257, 32, 32, 0, "pow2"),
    (2, 190, 128, 128, 0, "none"),
]


def _fp8_inputs(B, S, Hi, Di, ndocs, k_scale, seed):
    wl = synth.Workload("fp8", seed=seed, B=B, S=S, Hi=Hi, Di=Di, topk=4, H=1, Dqk=32, Dv=32,
                        backward=False, ndocs=ndocs)
    return wl, synth.indexer_inputs_fp8(wl, k_scale)


def _run_scores_fp8(inp):
    dsa = _dsa()
    seg = None if inp["seg"] is None else dev(inp["seg"])
    ks = None if inp["k_scale"] is None else dev(inp["k_scale"])
    sc = dsa.dsa_index_scores_fp8(dev(inp["q_idx"]), dev(inp["k_idx"]), dev(inp["w"]), seg, ks)
    assert dsa.dsa_get_last_device_error() == 0
    return sc


@pytest.mark.parametrize("case", FP8_CASES)
def test_index_scores_fp8_exact(case):
    B, S, Hi, Di, ndocs, k_scale = case
    _, inp = _fp8_inputs(B, S, Hi, Di, ndocs, k_scale, seed=300 + S)
    sc = host_f64(_run_scores_fp8(inp))
    ref = oracle.index_scores_fp8(inp["q_idx"], inp["k_idx"], inp["w"], inp["seg"], inp["k_scale"])
    _check_scores(sc, ref, np.arange(B * S), S)


def test_index_scores_fp8_equals_bf16_kernel():
    """The same dyadic values through both kernels: identical scores."""
    wl, f = _fp8_inputs(1, 611, 64, 128, 2, "none", seed=41)
    a = synth.indexer_inputs(wl)
    sc8 = host_f64(_run_scores_fp8(f))
    sc16 = host_f64(_run_scores(a))
    for t in range(611):
        assert np.array_equal(sc8[0, t, : t + 1], sc16[0, t, : t + 1]), t


def test_index_scores_fp8_general_key_scale():
    """Scales that are not powers of two: one fp32 rounding of the scaled (exact) sum."""
    B, S = 1, 400
    _, inp = _fp8_inputs(B, S, 64, 128, 0, "dyadic", seed=42)
    sc = host_f64(_run_scores_fp8(inp))
    ref = oracle.index_scores_fp8(inp["q_idx"], inp["k_idx"], inp["w"], None, inp["k_scale"])
    for t in range(S):
        g, o = sc[0, t, : t + 1], ref[t, : t + 1]
        assert np.all(np.abs(g - o) <= 2.0 ** -24 * np.abs(o)), t


def test_index_scores_fp8_rejects_wide_dtypes():
    dsa = _dsa()
    _, inp = _fp8_inputs(1, 64, 4, 32, 0, "none", seed=43)
    with pytest.raises(TypeError):
        dsa.dsa_index_scores_fp8(bf16_dev(synth.dyadic_bf16((1, 64, 4, 32), 1, 1, -8, 8, 3)),
                                 dev(inp["k_idx"]), dev(inp["w"]))


# ------------------------------------------------------------------- top-k

def _check_topk(idx_gpu, cnt_gpu, scores_f64, seg, S, k, rows):
    ref_idx, ref_cnt = oracle.topk(scores_f64, seg, S, k, rows=rows, B=idx_gpu.shape[0])
    flat_idx = idx_gpu.reshape(-1, k)[rows]
    flat_cnt = cnt_gpu.reshape(-1)[rows]
    for r in range(len(rows)):
        assert np.array_equal(flat_idx[r], ref_idx[r]), (int(rows[r]), flat_idx[r][:8],
                                                         ref_idx[r][:8])
    assert np.array_equal(flat_cnt, ref_cnt)


@pytest.mark.parametrize("case", INDEXER_CASES[:4])
@pytest.mark.parametrize("k", [1, 4, 37, 300])
def test_topk_on_gpu_scores_exact(case, k):
    dsa = _dsa()
    B, S, Hi, Di, ndocs, w_kind = case
    inp = _indexer_case(B, S, Hi, Di, seed=200 + S, ndocs=ndocs, w_kind=w_kind)
    sc = _run_scores(inp)
    seg = None if inp["seg"] is None else dev(inp["seg"])
    idx, cnt = dsa.dsa_topk(sc, k, seg)
    rows = np.arange(B * S)
    sc64 = host_f64(sc[:, :, :S]).reshape(B * S, S)
    _check_topk(idx.cpu().numpy(), cnt.cpu().numpy(), sc64, inp["seg"], S, k, rows)


@pytest.mark.parametrize("ndocs", [0, 3])
@pytest.mark.parametrize("k", [1, 2, 64, 999, 2000])
def test_topk_heavy_ties(ndocs, k):
    """Scores from a 7-value set with both zeros: ties decide most of the selection."""
    dsa = _dsa()
    B, S = 2, 1000
    rng = np.random.default_rng(ndocs * 100 + k)
    vals = np.array([-2.0, -0.5, -0.0, 0.0, 0.25, 0.25, 1.0], dtype=np.float32)
    sc = vals[rng.integers(0, len(vals), size=(B, S, S))]
    seg = synth.segments(B, S, ndocs, 9) if ndocs else None
    sct = dev(sc)
    idx, cnt = dsa.dsa_topk(sct, k, None if seg is None else dev(seg))
    _check_topk(idx.cpu().numpy(), cnt.cpu().numpy(), sc.reshape(B * S, S).astype(np.float64),
                seg, S, k, np.arange(B * S))


@pytest.mark.parametrize("kind", ["ulps", "wide"])
@pytest.mark.parametrize("k", [3, 100, 700])
def test_topk_close_and_wide_keys(kind, k):
    """Keys a few ulps apart (every radix digit decides) and keys over ~120 octaves
    (the k-th largest far below the row maximum)."""
    dsa = _dsa()
    B, S = 1, 900
    rng = np.random.default_rng(k + (0 if kind == "ulps" else 1))
    if kind == "ulps":
        base = np.float32(1.0 + 2.0 ** -10)
        sc = base + rng.integers(-300, 300, size=(B, S, S)).astype(np.float32) * np.float32(2 ** -23)
        sc[..., ::5] *= -1
    else:
        mant = rng.uniform(1.0, 2.0, size=(B, S, S))
        sc = (np.sign(rng.standard_normal((B, S, S))) * mant *
              np.exp2(rng.integers(-60, 61, size=(B, S, S)))).astype(np.float32)
        sc[0, :, 0] = 1e30   # one huge key per row
    idx, cnt = dsa.dsa_topk(dev(sc.astype(np.float32)), k)
    _check_topk(idx.cpu().numpy(), cnt.cpu().numpy(),
                sc.astype(np.float32).reshape(B * S, S).astype(np.float64), None, S, k,
                np.arange(B * S))


def test_topk_rows_longer_than_the_shared_stage():
    dsa = _dsa()
    S, k = 17000, 100
    rng = np.random.default_rng(3)
    sc = rng.standard_normal((1, S, S), dtype=np.float32)
    sc[0, -1, ::7] = 3.5   # ties at the top of the last row
    idx, cnt = dsa.dsa_topk(dev(sc), k)
    rows = np.array([0, 50, 16383, 16384, 16385, 16999], dtype=np.int64)
    _check_topk(idx.cpu().numpy(), cnt.cpu().numpy(), sc[0][rows].astype(np.float64), None, S,
                k, rows)


def test_topk_long_rows_two_batches():
    """Two batch rows past the shared stage: the persistent long-row CTAs take (batch, query)
    rows interleaved, longest first; sampled rows of both against the oracle, with each
    slot's selected score."""
    dsa = _dsa()
    B, S, k = 2, 17000, 100
    rng = np.random.default_rng(23)
    sc = rng.standard_normal((B, S, S), dtype=np.float32)
    sc[1, -1, ::5] = 2.75   # ties at the top of batch row 1's last query
    idx, cnt, vals = dsa.dsa_topk(dev(sc), k, vals=True)
    assert dsa.dsa_get_last_device_error() == 0
    rows = np.array([100, 16383, 16384, 16999, S + 16384, S + 16500, 2 * S - 1], dtype=np.int64)
    idx_h = idx.cpu().numpy()
    _check_topk(idx_h, cnt.cpu().numpy(), sc.reshape(B * S, S)[rows].astype(np.float64), None,
                S, k, rows)
    flat_idx = idx_h.reshape(B * S, k)
    flat_vals = vals.cpu().numpy().reshape(B * S, k)
    for r in rows:
        sel = flat_idx[r]
        want = np.where(sel >= 0, sc.reshape(B * S, S)[r, np.maximum(sel, 0)], -np.inf)
        assert np.array_equal(flat_vals[r], want.astype(np.float32))


def test_topk_long_rows_k2048():
    """Rows of 16384 to 32767 keys with k = 2048, the long-context regime of the long-row
    kernel's one-pass path (thousands of candidates per row): sampled rows against the oracle."""
    dsa = _dsa()
    S, k = 32768, 2048
    rng = np.random.default_rng(11)
    sc = rng.standard_normal((1, S, S), dtype=np.float32)
    idx, cnt = dsa.dsa_topk(dev(sc), k)
    assert dsa.dsa_get_last_device_error() == 0
    rows = np.array([16383, 16384, 16385, 20000, 24575, 28000, 32767], dtype=np.int64)
    _check_topk(idx.cpu().numpy(), cnt.cpu().numpy(), sc[0][rows].astype(np.float64), None, S,
                k, rows)


def test_topk_long_rows_with_segments():
    """Rows longer than the shared stage with packed documents: the long-row kernel with its
    per-key segment test (its whole-group fast path applies only without segment ids), and
    rows whose document is shorter than k."""
    dsa = _dsa()
    S, k = 20000, 300
    rng = np.random.default_rng(12)
    sc = rng.standard_normal((1, S, S), dtype=np.float32)
    # documents [0, 9000), [9000, 19800), [19800, 20000): the last one holds 200 < k keys and
    # its rows lie beyond the staged kernel's 16384 keys
    seg = np.zeros((1, S), dtype=np.int32)
    seg[0, 9000:] = 1
    seg[0, 19800:] = 2
    idx, cnt = dsa.dsa_topk(dev(sc), k, dev(seg))
    assert dsa.dsa_get_last_device_error() == 0
    rows = np.array([16383, 16384, 16385, 18000, 19799, 19800, 19850, S - 1], dtype=np.int64)
    short = [r for r in rows if r - 19800 + 1 < k and r >= 19800]
    assert len(short) == 3 and min(short) >= 16384
    _check_topk(idx.cpu().numpy(), cnt.cpu().numpy(), sc[0][rows].astype(np.float64), seg, S,
                k, rows)
    got = cnt.cpu().numpy()[0]
    assert [int(got[r]) for r in short] == [r - 19800 + 1 for r in short]


def test_topk_long_rows_ties_two_pass():
    """Long rows whose candidate list cannot settle them in one pass: a row of equal scores
    (every key a candidate), a row with 4 distinct values (about 5000 keys tied at the
    threshold), a row of +0 and -0 only, and a row with half its keys tied at 1.0 above
    normal noise. The long-row kernel takes its two-pass path for these; neighbouring rows
    of plain noise take the one-pass path in the same launch."""
    dsa = _dsa()
    S, k = 20000, 2048
    rng = np.random.default_rng(21)
    sc = rng.standard_normal((1, S, S), dtype=np.float32)
    sc[0, 17000, :] = 0.25
    sc[0, 18000, :] = rng.integers(0, 4, S).astype(np.float32)
    sc[0, 19000, :] = np.where(rng.random(S) < 0.5, np.float32(0.0), np.float32(-0.0))
    sc[0, 19999, :] = np.where(rng.random(S) < 0.5, np.float32(1.0),
                               np.minimum(rng.standard_normal(S).astype(np.float32), 0.9))
    idx, cnt, vals = dsa.dsa_topk(dev(sc), k, vals=True)
    assert dsa.dsa_get_last_device_error() == 0
    rows = np.array([16999, 17000, 17001, 18000, 19000, 19998, 19999], dtype=np.int64)
    idx_h = idx.cpu().numpy()
    _check_topk(idx_h, cnt.cpu().numpy(), sc[0][rows].astype(np.float64), None, S, k, rows)
    # each slot's score is the row's score at the selected key (bit for bit; -0 stays -0)
    vals_h = vals.cpu().numpy().reshape(S, k)[rows]
    for r, t in enumerate(rows):
        sel = idx_h[0, t]
        assert np.all(sel >= 0)
        assert np.array_equal(vals_h[r].view(np.uint32), sc[0, t, sel].view(np.uint32))


def test_topk_golden_fixtures_on_gpu():
    from test_oracle_pins import _parse_golden
    dsa = _dsa()
    for k, seg, scores, expect in _parse_golden():
        S = len(scores)
        sc = np.zeros((1, S, (S + 3) // 4 * 4), dtype=np.float32)
        sc[0, S - 1, :S] = scores
        segt = None if seg is None else dev(np.array([seg], dtype=np.int32))
        idx, cnt = dsa.dsa_topk(dev(sc), k, segt, S=S)
        assert idx[0, S - 1].cpu().tolist() == expect


# --------------------------------------------------------------- attention

ATTN_CASES = [
    # B, S, H, Dqk, Dv, k, ndocs
    (1, 128, 2, 32, 32, 4, 0),
    (1, 489, 16, 192, 128, 512, 3),
    (1, 300, 128, 192, 128, 64, 0),
    (2, 200, 16, 192, 128, 100, 0),
    (1, 150, 64, 128, 128, 40, 0),
    (1, 130, 32, 64, 64, 33, 2),
    (1, 100, 8, 192, 128, 7, 0),
    (1, 96, 128, 192, 128, 200, 0),
    (1, 260, 128, 128, 128, 150, 0),
    (1, 200, 96, 192, 128, 97, 2),
    (2, 150, 128, 192, 128, 300, 0),
    (1, 700, 128, 192, 128, 512, 3),
    # few heads on the tensor-core kernels (TMEM lanes >= H idle)
    (1, 333, 1, 192, 128, 100, 0),
    (2, 177, 3, 192, 128, 61, 2),
    (1, 210, 5, 128, 128, 96, 0),
]


def _attn_case(B, S, H, Dqk, Dv, k, ndocs, seed):
    Q = synth.normal_bf16((B, S, H, Dqk), seed, synth.STREAM_Q)
    K = synth.normal_bf16((B, S, 1, Dqk), seed, synth.STREAM_K)
    V = synth.normal_bf16((B, S, 1, Dv), seed, synth.STREAM_V)
    dO = synth.normal_bf16((B, S, H, Dv), seed, synth.STREAM_DO)
    ind = _indexer_case(B, S, 4, 32, seed, ndocs=ndocs)
    sc = oracle.index_scores(ind["q_idx"], ind["k_idx"], ind["w"], ind["seg"])
    idx, _ = oracle.topk(sc, ind["seg"], S, k, B=B)
    return Q, K, V, dO, idx.reshape(B, S, k)


@pytest.mark.parametrize("case", ATTN_CASES)
def test_sparse_attn_fwd_bwd(case):
    dsa = _dsa()
    B, S, H, Dqk, Dv, k, ndocs = case
    Q, K, V, dO, idx = _attn_case(*case, seed=300 + S + H)
    scale = 1.0 / np.sqrt(Dqk)
    Qd, Kd, Vd, dOd, idxd = bf16_dev(Q), bf16_dev(K), bf16_dev(V), bf16_dev(dO), dev(idx)
    O, lse = dsa.dsa_sparse_attn_fwd(Qd, Kd, Vd, idxd, scale)
    dQ, dK, dV = dsa.dsa_sparse_attn_bwd(Qd, Kd, Vd, idxd, O, lse, dOd, scale)
    assert dsa.dsa_get_last_device_error() == 0
    O_ref, lse_ref = oracle.attn_fwd(Q, K, V, idx, scale)
    assert rel_err(host_f64(O).reshape(O_ref.shape), O_ref) <= TOL
    assert rel_err(host_f64(lse).reshape(lse_ref.shape), lse_ref) <= TOL
    dQ_ref, dK_ref, dV_ref = oracle.attn_bwd(Q, K, V, idx, dO, scale)
    assert rel_err(host_f64(dQ).reshape(dQ_ref.shape), dQ_ref) <= TOL
    assert rel_err(host_f64(dK), dK_ref) <= TOL
    assert rel_err(host_f64(dV), dV_ref) <= TOL


@pytest.mark.parametrize("H", [16, 128])
def test_sparse_attn_user_index_lists(H):
    """-1 anywhere, entries above the diagonal, empty rows, unsorted lists."""
    dsa = _dsa()
    B, S, Dqk, Dv, k = 1, 80, 192, 128, 70
    Q, K, V, dO, _ = _attn_case(B, S, H, Dqk, Dv, 8, 0, seed=5)
    rng = np.random.default_rng(11)
    idx = np.full((B, S, k), -1, dtype=np.int32)
    for t in range(S):
        if t % 9 == 4:
            continue                                    # empty row
        pick = rng.choice(S, size=min(S, k), replace=False).astype(np.int32)
        pick[rng.random(pick.size) < 0.2] = -1          # holes
        idx[0, t] = pick                                # some above the diagonal
    scale = 0.1
    Qd, Kd, Vd, dOd, idxd = bf16_dev(Q), bf16_dev(K), bf16_dev(V), bf16_dev(dO), dev(idx)
    O, lse = dsa.dsa_sparse_attn_fwd(Qd, Kd, Vd, idxd, scale)
    dQ, dK, dV = dsa.dsa_sparse_attn_bwd(Qd, Kd, Vd, idxd, O, lse, dOd, scale)
    assert dsa.dsa_get_last_device_error() == 0
    O_ref, lse_ref = oracle.attn_fwd(Q, K, V, idx, scale)
    assert rel_err(host_f64(O).reshape(O_ref.shape), O_ref) <= TOL
    lg = host_f64(lse).reshape(lse_ref.shape)
    assert np.array_equal(np.isneginf(lg), np.isneginf(lse_ref))
    fin = np.isfinite(lse_ref)
    assert rel_err(lg[fin], lse_ref[fin]) <= TOL
    dQ_ref, dK_ref, dV_ref = oracle.attn_bwd(Q, K, V, idx, dO, scale)
    assert rel_err(host_f64(dQ).reshape(dQ_ref.shape), dQ_ref) <= TOL
    assert rel_err(host_f64(dK), dK_ref) <= TOL
    assert rel_err(host_f64(dV), dV_ref) <= TOL


# ------------------------------------------------- dense-tile forward kernel

DENSE_CASES = [
    # B, S, H, Dqk, Dv, k, ndocs
    (1, 489, 16, 192, 128, 512, 3),
    (2, 200, 16, 192, 128, 100, 0),
    (1, 129, 1, 192, 128, 64, 0),      # the last query tile holds one row
    (1, 300, 128, 192, 128, 64, 0),    # many heads (the call would pick the other kernel)
    (1, 260, 8, 128, 128, 300, 0),     # k >= S: every causal key
    (2, 177, 3, 192, 128, 61, 2),
    (1, 700, 16, 192, 128, 96, 0),     # many skipped key tiles
]


def _fwd_check(O, lse, Q, K, V, idx, scale):
    O_ref, lse_ref = oracle.attn_fwd(Q, K, V, idx, scale)
    assert rel_err(host_f64(O).reshape(O_ref.shape), O_ref) <= TOL
    lg = host_f64(lse).reshape(lse_ref.shape)
    assert np.array_equal(np.isneginf(lg), np.isneginf(lse_ref))
    fin = np.isfinite(lse_ref)
    assert rel_err(lg[fin], lse_ref[fin]) <= TOL


@pytest.mark.parametrize("case", DENSE_CASES)
def test_dense_fwd_matches_oracle(case):
    dsa = _dsa()
    B, S, H, Dqk, Dv, k, ndocs = case
    Q, K, V, dO, idx = _attn_case(*case, seed=900 + S + H)
    scale = 1.0 / np.sqrt(Dqk)
    O, lse = dsa.dsa_sparse_attn_fwd_dense(bf16_dev(Q), bf16_dev(K), bf16_dev(V), dev(idx), scale)
    assert dsa.dsa_get_last_device_error() == 0
    _fwd_check(O, lse, Q, K, V, idx, scale)


@pytest.mark.parametrize("H", [16, 128])
def test_dense_fwd_user_index_lists(H):
    """-1 anywhere, entries above the diagonal, empty rows, unsorted lists."""
    dsa = _dsa()
    B, S, Dqk, Dv, k = 1, 300, 192, 128, 150
    Q, K, V, dO, _ = _attn_case(B, S, H, Dqk, Dv, 8, 0, seed=15)
    rng = np.random.default_rng(12)
    idx = np.full((B, S, k), -1, dtype=np.int32)
    for t in range(S):
        if t % 9 == 4 or 128 <= t < 140:
            continue                                    # empty rows
        pick = rng.choice(S, size=min(S, k), replace=False).astype(np.int32)
        pick[rng.random(pick.size) < 0.2] = -1          # holes
        idx[0, t] = pick                                # some above the diagonal
    O, lse = dsa.dsa_sparse_attn_fwd_dense(bf16_dev(Q), bf16_dev(K), bf16_dev(V), dev(idx), 0.1)
    assert dsa.dsa_get_last_device_error() == 0
    _fwd_check(O, lse, Q, K, V, idx, 0.1)


def test_dense_fwd_query_tile_without_keys():
    """A whole query tile that selects nothing: O = 0, LSE = -inf, the others unaffected."""
    dsa = _dsa()
    B, S, H, k = 1, 300, 4, 32
    Q, K, V, dO, idx = _attn_case(B, S, H, 192, 128, k, 0, seed=16)
    idx = idx.copy()
    idx[0, 128:256] = -1
    O, lse = dsa.dsa_sparse_attn_fwd_dense(bf16_dev(Q), bf16_dev(K), bf16_dev(V), dev(idx), 0.07)
    assert dsa.dsa_get_last_device_error() == 0
    _fwd_check(O, lse, Q, K, V, idx, 0.07)
    assert torch.all(O[0, 128:256] == 0)


def _bwd_check(dQ, dK, dV, Q, K, V, idx, dO, scale):
    dQ_ref, dK_ref, dV_ref = oracle.attn_bwd(Q, K, V, idx, dO, scale)
    assert rel_err(host_f64(dQ).reshape(dQ_ref.shape), dQ_ref) <= TOL
    assert rel_err(host_f64(dK), dK_ref) <= TOL
    assert rel_err(host_f64(dV), dV_ref) <= TOL


@pytest.mark.parametrize("case", DENSE_CASES)
def test_dense_bwd_matches_oracle(case):
    dsa = _dsa()
    B, S, H, Dqk, Dv, k, ndocs = case
    Q, K, V, dO, idx = _attn_case(*case, seed=950 + S + H)
    scale = 1.0 / np.sqrt(Dqk)
    Qd, Kd, Vd, dOd, idxd = bf16_dev(Q), bf16_dev(K), bf16_dev(V), bf16_dev(dO), dev(idx)
    O, lse = dsa.dsa_sparse_attn_fwd(Qd, Kd, Vd, idxd, scale)
    dQ, dK, dV = dsa.dsa_sparse_attn_bwd_dense(Qd, Kd, Vd, idxd, O, lse, dOd, scale)
    assert dsa.dsa_get_last_device_error() == 0
    _bwd_check(dQ, dK, dV, Q, K, V, idx, dO, scale)


@pytest.mark.parametrize("H", [5, 16])
def test_dense_bwd_user_lists_and_empty_tiles(H):
    """Holes, entries above the diagonal, empty rows and a whole query tile without keys;
    H = 5 leaves a partial group of heads in the dK / dV pass."""
    dsa = _dsa()
    B, S, Dqk, Dv, k = 1, 300, 192, 128, 150
    Q, K, V, dO, _ = _attn_case(B, S, H, Dqk, Dv, 8, 0, seed=21)
    rng = np.random.default_rng(22)
    idx = np.full((B, S, k), -1, dtype=np.int32)
    for t in range(S):
        if t % 9 == 4 or 128 <= t < 256:
            continue
        pick = rng.choice(S, size=min(S, k), replace=False).astype(np.int32)
        pick[rng.random(pick.size) < 0.2] = -1
        idx[0, t] = pick
    Qd, Kd, Vd, dOd, idxd = bf16_dev(Q), bf16_dev(K), bf16_dev(V), bf16_dev(dO), dev(idx)
    O, lse = dsa.dsa_sparse_attn_fwd(Qd, Kd, Vd, idxd, 0.1)
    dQ, dK, dV = dsa.dsa_sparse_attn_bwd_dense(Qd, Kd, Vd, idxd, O, lse, dOd, 0.1)
    assert dsa.dsa_get_last_device_error() == 0
    _bwd_check(dQ, dK, dV, Q, K, V, idx, dO, 0.1)
    assert torch.all(dQ[0, 128:256] == 0)


def test_bwd_kernel_choice():
    dsa = _dsa()
    sc = 1.0 / np.sqrt(192)
    assert dsa.dsa_sparse_attn_bwd_kernel(4, 4096, 16, 1, 192, 128, 512, sc) == dsa.DSA_BWD_DENSE_TC
    assert dsa.dsa_sparse_attn_bwd_kernel(1, 16384, 128, 1, 192, 128, 2048, sc) == \
        dsa.DSA_BWD_GATHER_TC
    assert dsa.dsa_sparse_attn_bwd_kernel(1, 128, 2, 1, 32, 32, 4, 0.2) == dsa.DSA_BWD_MMA_SYNC


def test_fwd_kernel_choice():
    """The automatic forward picks the dense-tile kernel for few heads and many selected keys,
    the gathered-key kernel for 128 heads, mma.sync for small head dims; Hkv > 1 always
    takes the dense-tile kernel, and is refused where that kernel does not apply."""
    dsa = _dsa()
    sc = 1.0 / np.sqrt(192)
    assert dsa.dsa_sparse_attn_fwd_kernel(2, 4096, 16, 1, 192, 128, 2048, sc) == dsa.DSA_FWD_DENSE_TC
    assert dsa.dsa_sparse_attn_fwd_kernel(4, 4096, 16, 1, 192, 128, 512, sc) == dsa.DSA_FWD_DENSE_TC
    assert dsa.dsa_sparse_attn_fwd_kernel(1, 16384, 128, 1, 192, 128, 2048, sc) == \
        dsa.DSA_FWD_GATHER_TC
    assert dsa.dsa_sparse_attn_fwd_kernel(1, 489, 16, 1, 192, 128, 512, sc) == \
        dsa.DSA_FWD_GATHER_TC   # too few work items to fill the GPU
    assert dsa.dsa_sparse_attn_fwd_kernel(1, 128, 2, 1, 32, 32, 4, 0.2) == dsa.DSA_FWD_MMA_SYNC
    assert dsa.dsa_sparse_attn_fwd_kernel(1, 128, 2, 2, 192, 128, 4, 0.2) == dsa.DSA_FWD_DENSE_TC
    with pytest.raises(dsa.DsaError):
        dsa.dsa_sparse_attn_fwd_kernel(1, 128, 2, 2, 32, 32, 4, 0.2)


def test_dense_fwd_bad_index_and_unsupported():
    dsa = _dsa()
    B, S, H, k = 1, 140, 16, 8
    Q, K, V, dO, idx = _attn_case(B, S, H, 192, 128, k, 0, seed=17)
    idx = idx.copy()
    idx[0, 100, 0] = S + 3      # out of range: skipped and reported
    dsa.dsa_get_last_device_error()
    O, lse = dsa.dsa_sparse_attn_fwd_dense(bf16_dev(Q), bf16_dev(K), bf16_dev(V), dev(idx), 0.125)
    assert dsa.dsa_get_last_device_error() == (0x300 | 0x02)
    idx_ok = idx.copy()
    idx_ok[0, 100, 0] = -1
    _fwd_check(O, lse, Q, K, V, idx_ok, 0.125)
    Q6, K6, V6, _, idx6 = _attn_case(1, 64, 4, 64, 64, 8, 0, seed=18)
    with pytest.raises(dsa.DsaError):
        dsa.dsa_sparse_attn_fwd_dense(bf16_dev(Q6), bf16_dev(K6), bf16_dev(V6), dev(idx6), 0.125)


def test_bad_index_is_reported_not_faulted():
    dsa = _dsa()
    B, S, H, D, k = 1, 40, 16, 64, 8
    Q, K, V, dO, idx = _attn_case(B, S, H, D, D, k, 0, seed=6)
    idx = idx.copy()
    idx[0, 30, 0] = S + 5      # out of range: skipped and reported
    Qd, Kd, Vd = bf16_dev(Q), bf16_dev(K), bf16_dev(V)
    dsa.dsa_get_last_device_error()
    O, lse = dsa.dsa_sparse_attn_fwd(Qd, Kd, Vd, dev(idx), 0.125)
    code = dsa.dsa_get_last_device_error()
    assert code == (0x300 | 0x02)
    assert dsa.dsa_get_last_device_error() == 0   # cleared by the read
    idx_ok = idx.copy()
    idx_ok[0, 30, 0] = -1
    O_ref, _ = oracle.attn_fwd(Q, K, V, idx_ok, 0.125)
    assert rel_err(host_f64(O).reshape(O_ref.shape), O_ref) <= TOL


# ------------------------------------- per-head and grouped K / V (Hkv > 1)

HKV_CASES = [
    # B, S, H, Hkv, Dqk, Dv, k, ndocs
    (1, 300, 16, 16, 192, 128, 64, 0),     # one K / V head per query head
    (2, 200, 8, 2, 192, 128, 100, 0),      # groups of four heads
    (1, 260, 4, 4, 128, 128, 300, 0),      # k >= S: every causal key
    (1, 489, 16, 4, 192, 128, 512, 3),     # packed documents, ragged last tile
    (1, 129, 2, 2, 192, 128, 64, 0),
    (1, 200, 128, 128, 192, 128, 100, 0),  # 128 heads, each with its own K / V
]


def _hkv_case(B, S, H, Hkv, Dqk, Dv, k, ndocs, seed):
    Q = synth.normal_bf16((B, S, H, Dqk), seed, synth.STREAM_Q)
    K = synth.normal_bf16((B, S, Hkv, Dqk), seed, synth.STREAM_K)
    V = synth.normal_bf16((B, S, Hkv, Dv), seed, synth.STREAM_V)
    dO = synth.normal_bf16((B, S, H, Dv), seed, synth.STREAM_DO)
    ind = _indexer_case(B, S, 4, 32, seed, ndocs=ndocs)
    sc = oracle.index_scores(ind["q_idx"], ind["k_idx"], ind["w"], ind["seg"])
    idx, _ = oracle.topk(sc, ind["seg"], S, k, B=B)
    return Q, K, V, dO, idx.reshape(B, S, k)


@pytest.mark.parametrize("case", HKV_CASES)
def test_per_head_kv_fwd_bwd(case):
    dsa = _dsa()
    B, S, H, Hkv, Dqk, Dv, k, ndocs = case
    Q, K, V, dO, idx = _hkv_case(*case, seed=900 + S + H + Hkv)
    scale = 1.0 / np.sqrt(Dqk)
    assert dsa.dsa_sparse_attn_fwd_kernel(B, S, H, Hkv, Dqk, Dv, k, scale) == dsa.DSA_FWD_DENSE_TC
    assert dsa.dsa_sparse_attn_bwd_kernel(B, S, H, Hkv, Dqk, Dv, k, scale) == dsa.DSA_BWD_DENSE_TC
    Qd, Kd, Vd, dOd, idxd = bf16_dev(Q), bf16_dev(K), bf16_dev(V), bf16_dev(dO), dev(idx)
    O, lse = dsa.dsa_sparse_attn_fwd(Qd, Kd, Vd, idxd, scale)
    dQ, dK, dV = dsa.dsa_sparse_attn_bwd(Qd, Kd, Vd, idxd, O, lse, dOd, scale)
    assert dsa.dsa_get_last_device_error() == 0
    O_ref, lse_ref = oracle.attn_fwd(Q, K, V, idx, scale)
    assert rel_err(host_f64(O).reshape(O_ref.shape), O_ref) <= TOL
    assert rel_err(host_f64(lse).reshape(lse_ref.shape), lse_ref) <= TOL
    dQ_ref, dK_ref, dV_ref = oracle.attn_bwd(Q, K, V, idx, dO, scale)
    assert rel_err(host_f64(dQ).reshape(dQ_ref.shape), dQ_ref) <= TOL
    assert rel_err(host_f64(dK), dK_ref) <= TOL
    assert rel_err(host_f64(dV), dV_ref) <= TOL
    # each K / V head's gradient on its own (a mix-up of heads would hide in the max norm)
    for g in range(Hkv):
        assert rel_err(host_f64(dK)[:, :, g], dK_ref[:, :, g]) <= TOL
        assert rel_err(host_f64(dV)[:, :, g], dV_ref[:, :, g]) <= TOL


def test_per_head_kv_user_lists():
    """-1 holes, entries above the diagonal and empty rows with Hkv = H."""
    dsa = _dsa()
    B, S, H, Hkv, Dqk, Dv, k = 1, 150, 8, 8, 192, 128, 60
    Q, K, V, dO, _ = _hkv_case(B, S, H, Hkv, Dqk, Dv, 8, 0, seed=77)
    rng = np.random.default_rng(19)
    idx = np.full((B, S, k), -1, dtype=np.int32)
    for t in range(S):
        if t % 13 == 5:
            continue
        pick = rng.choice(S, size=k, replace=False).astype(np.int32)
        pick[rng.random(k) < 0.25] = -1
        idx[0, t] = pick
    scale = 0.09
    Qd, Kd, Vd, dOd, idxd = bf16_dev(Q), bf16_dev(K), bf16_dev(V), bf16_dev(dO), dev(idx)
    O, lse = dsa.dsa_sparse_attn_fwd(Qd, Kd, Vd, idxd, scale)
    dQ, dK, dV = dsa.dsa_sparse_attn_bwd(Qd, Kd, Vd, idxd, O, lse, dOd, scale)
    assert dsa.dsa_get_last_device_error() == 0
    O_ref, lse_ref = oracle.attn_fwd(Q, K, V, idx, scale)
    assert rel_err(host_f64(O).reshape(O_ref.shape), O_ref) <= TOL
    lg = host_f64(lse).reshape(lse_ref.shape)
    assert np.array_equal(np.isneginf(lg), np.isneginf(lse_ref))
    dQ_ref, dK_ref, dV_ref = oracle.attn_bwd(Q, K, V, idx, dO, scale)
    assert rel_err(host_f64(dQ).reshape(dQ_ref.shape), dQ_ref) <= TOL
    assert rel_err(host_f64(dK), dK_ref) <= TOL
    assert rel_err(host_f64(dV), dV_ref) <= TOL


def test_per_head_kv_unsupported_forms():
    """Hkv > 1 needs the dense-tile kernels: other dims, the no-allocation backward and a
    head count that Hkv does not divide are refused before anything runs."""
    dsa = _dsa()
    with pytest.raises(dsa.DsaError) as e:
        dsa.dsa_sparse_attn_fwd_kernel(1, 64, 4, 2, 64, 64, 8, 0.1)
    assert e.value.status == dsa.DSA_ERR_UNSUPPORTED
    with pytest.raises(dsa.DsaError) as e:
        dsa.dsa_sparse_attn_bwd_kernel(1, 64, 6, 4, 192, 128, 8, 0.1)
    assert e.value.status == dsa.DSA_ERR_INVALID_ARG
    B, S, H, Hkv, Dqk, Dv, k = 1, 64, 4, 2, 192, 128, 8
    Q, K, V, dO, idx = _hkv_case(B, S, H, Hkv, Dqk, Dv, k, 0, seed=5)
    Qd, Kd, Vd, dOd, idxd = bf16_dev(Q), bf16_dev(K), bf16_dev(V), bf16_dev(dO), dev(idx)
    O, lse = dsa.dsa_sparse_attn_fwd(Qd, Kd, Vd, idxd, 0.1)
    with pytest.raises(dsa.DsaError) as e:
        dsa.dsa_sparse_attn_bwd_noalloc(Qd, Kd, Vd, idxd, O, lse, dOd, 0.1)
    assert e.value.status == dsa.DSA_ERR_UNSUPPORTED
    assert dsa.dsa_get_last_device_error() == 0


# --------------------------------------- fused indexer + top-k by query blocks

@pytest.mark.parametrize("case", [
    # B, S, Hi, Di, k, ndocs, block_rows
    (2, 700, 64, 128, 64, 0, 256),     # three full blocks and a ragged one
    (1, 700, 64, 128, 300, 3, 512),    # packed documents, k larger than early rows
    (1, 333, 4, 32, 100, 0, 256),      # 64 queries per indexer tile
    (1, 200, 16, 64, 8, 0, 2048),      # one block larger than S
    (1, 2000, 4, 32, 64, 0, 256),      # eight blocks through one reused buffer
    (2, 1500, 4, 32, 200, 3, 256),
])
def test_index_topk_matches_oracle(case):
    dsa = _dsa()
    B, S, Hi, Di, k, ndocs, R = case
    inp = _indexer_case(B, S, Hi, Di, seed=610 + S + Hi, ndocs=ndocs)
    seg = None if inp["seg"] is None else dev(inp["seg"])
    idx, cnt = dsa.dsa_index_topk(bf16_dev(inp["q_idx"]), bf16_dev(inp["k_idx"]), dev(inp["w"]),
                                  k, seg, block_rows=R)
    assert dsa.dsa_get_last_device_error() == 0
    sc = oracle.index_scores(inp["q_idx"], inp["k_idx"], inp["w"], inp["seg"])
    ref_idx, ref_cnt = oracle.topk(sc, inp["seg"], S, k, B=B)
    assert np.array_equal(idx.cpu().numpy().reshape(-1, k), ref_idx)
    assert np.array_equal(cnt.cpu().numpy().reshape(-1), ref_cnt)


def test_index_topk_long_rows_match_unfused_path():
    """S = 20000 crosses the 16384-key boundary of the staged top-k inside a block: the fused
    call equals the unfused path bit for bit, and the oracle on rows around the boundary."""
    dsa = _dsa()
    B, S, Hi, Di, k, R = 1, 20000, 64, 128, 2048, 4096
    inp = _indexer_case(B, S, Hi, Di, seed=77)
    q, kk, w = bf16_dev(inp["q_idx"]), bf16_dev(inp["k_idx"]), dev(inp["w"])
    idx_f, cnt_f = dsa.dsa_index_topk(q, kk, w, k, block_rows=R)
    scores = dsa.dsa_index_scores(q, kk, w)
    idx_u, cnt_u = dsa.dsa_topk(scores, k)
    assert dsa.dsa_get_last_device_error() == 0
    assert torch.equal(idx_f, idx_u) and torch.equal(cnt_f, cnt_u)
    rows = np.array([0, 2047, 2048, 4095, 4096, 16383, 16384, 16385, 19999], dtype=np.int64)
    sc = oracle.index_scores(inp["q_idx"], inp["k_idx"], inp["w"], None, rows=rows)
    ref_idx, ref_cnt = oracle.topk(sc, None, S, k, rows=rows, B=B)
    assert np.array_equal(idx_f.cpu().numpy().reshape(-1, k)[rows], ref_idx)
    assert np.array_equal(cnt_f.cpu().numpy().reshape(-1)[rows], ref_cnt)


@pytest.mark.parametrize("case", [
    # B, S, Hi, Di, k, ndocs, k_scale, block_rows
    (2, 700, 64, 128, 64, 0, "pow2", 256),
    (1, 489, 64, 128, 200, 3, "pow2", 256),
    (1, 1000, 8, 64, 100, 2, "none", 512),
])
def test_index_topk_fp8_matches_oracle(case):
    """The e4m3 indexer through query blocks: the oracle's e4m3 scores, then its top-k."""
    dsa = _dsa()
    B, S, Hi, Di, k, ndocs, k_scale, R = case
    _, inp = _fp8_inputs(B, S, Hi, Di, ndocs, k_scale, seed=640 + S)
    seg = None if inp["seg"] is None else dev(inp["seg"])
    ks = None if inp["k_scale"] is None else dev(inp["k_scale"])
    idx, cnt = dsa.dsa_index_topk(dev(inp["q_idx"]), dev(inp["k_idx"]), dev(inp["w"]), k, seg,
                                  block_rows=R, k_scale=ks)
    assert dsa.dsa_get_last_device_error() == 0
    sc = oracle.index_scores_fp8(inp["q_idx"], inp["k_idx"], inp["w"], inp["seg"], inp["k_scale"])
    ref_idx, ref_cnt = oracle.topk(sc, inp["seg"], S, k, B=B)
    assert np.array_equal(idx.cpu().numpy().reshape(-1, k), ref_idx)
    assert np.array_equal(cnt.cpu().numpy().reshape(-1), ref_cnt)


# ------------------------------- fused indexer + top-k, streaming form (no score rows)

@pytest.mark.parametrize("case", [
    # B, S, Hi, Di, k, ndocs, block_rows
    (1, 128, 4, 32, 4, 0, 256),        # the tiny workload's shape: every tile sampled
    (2, 3000, 64, 128, 300, 0, 512),   # rows past 16 tiles: a sampled window per row
    (1, 2500, 64, 128, 2048, 0, 256),  # k near the row length
    (2, 2000, 16, 64, 100, 3, 512),    # packed documents: windows from an estimated count
    (1, 489, 64, 128, 512, 3, 256),    # every row has at most k keys
    (1, 4100, 4, 32, 64, 0, 1024),     # 64 queries per indexer tile
    (1, 2300, 32, 32, 200, 0, 512),    # 4 queries per epilogue warp, listed per tile
    (1, 1500, 128, 128, 100, 2, 512),  # one query per epilogue warp, packed documents
    (1, 1800, 8, 64, 150, 0, 512),     # 32 queries per tile: list counters in global memory
    (1, 1200, 1, 64, 50, 0, 256),      # one head: 256 queries per tile
])
def test_index_topk_stream_matches_oracle(case):
    """The streaming form (sampled window, candidate lists, no score row) against the oracle's
    top-k of the oracle's scores, every row, bit for bit."""
    dsa = _dsa()
    B, S, Hi, Di, k, ndocs, R = case
    inp = _indexer_case(B, S, Hi, Di, seed=820 + S + Hi, ndocs=ndocs)
    seg = None if inp["seg"] is None else dev(inp["seg"])
    idx, cnt = dsa.dsa_index_topk_stream(bf16_dev(inp["q_idx"]), bf16_dev(inp["k_idx"]),
                                         dev(inp["w"]), k, seg, block_rows=R)
    assert dsa.dsa_get_last_device_error() == 0
    sc = oracle.index_scores(inp["q_idx"], inp["k_idx"], inp["w"], inp["seg"])
    ref_idx, ref_cnt = oracle.topk(sc, inp["seg"], S, k, B=B)
    assert np.array_equal(idx.cpu().numpy().reshape(-1, k), ref_idx)
    assert np.array_equal(cnt.cpu().numpy().reshape(-1), ref_cnt)


def test_index_topk_stream_matches_unfused_path_at_v32_shape():
    """The V3.2 indexer shape at S = 6000 with top-2048 (the bench's distribution of scores):
    the streaming form equals the unfused indexer + top-k on every row."""
    dsa = _dsa()
    wl = synth.WORKLOADS["v32_671b_s16k"].replace(S=6000)
    ind = synth.indexer_inputs(wl)
    q, kk, w = bf16_dev(ind["q_idx"]), bf16_dev(ind["k_idx"]), dev(ind["w"])
    idx_s, cnt_s = dsa.dsa_index_topk_stream(q, kk, w, wl.topk)
    idx_u, cnt_u = dsa.dsa_topk(dsa.dsa_index_scores(q, kk, w), wl.topk)
    assert dsa.dsa_get_last_device_error() == 0
    assert torch.equal(idx_s, idx_u) and torch.equal(cnt_s, cnt_u)


@pytest.mark.parametrize("S", [6000, 20000])
def test_index_topk_stream_rows_left_to_the_memory_form(S):
    """Every score equal: each row's window holds all its keys, so every row with more than
    4096 keys overflows the window list and is left unsettled; its block is redone by the
    memory form (gated on the device), across the 16384-key boundary for S = 20000. The
    selection is then the k lowest indices."""
    dsa = _dsa()
    B, Hi, Di, k = 1, 64, 128, 100
    one = torch.full((B, S, Hi, Di), 0.125, dtype=torch.bfloat16, device="cuda")
    kk = torch.full((B, S, Di), 0.125, dtype=torch.bfloat16, device="cuda")
    w = torch.full((B, S, Hi), 0.0625, dtype=torch.float32, device="cuda")
    idx, cnt = dsa.dsa_index_topk_stream(one, kk, w, k, block_rows=2048)
    assert dsa.dsa_get_last_device_error() == 0
    t = np.arange(S)
    ref = np.where(np.arange(k)[None, :] <= t[:, None], np.arange(k)[None, :], -1)
    assert np.array_equal(idx.cpu().numpy().reshape(S, k), ref)
    assert np.array_equal(cnt.cpu().numpy().reshape(S), np.minimum(t + 1, k))


def test_index_topk_stream_fp8_matches_oracle():
    dsa = _dsa()
    B, S, Hi, Di, k, ndocs = 1, 2600, 64, 128, 256, 2
    _, inp = _fp8_inputs(B, S, Hi, Di, ndocs, "pow2", seed=870)
    seg = dev(inp["seg"])
    idx, cnt = dsa.dsa_index_topk_stream(dev(inp["q_idx"]), dev(inp["k_idx"]), dev(inp["w"]), k,
                                         seg, block_rows=512, k_scale=dev(inp["k_scale"]))
    assert dsa.dsa_get_last_device_error() == 0
    sc = oracle.index_scores_fp8(inp["q_idx"], inp["k_idx"], inp["w"], inp["seg"], inp["k_scale"])
    ref_idx, ref_cnt = oracle.topk(sc, inp["seg"], S, k, B=B)
    assert np.array_equal(idx.cpu().numpy().reshape(-1, k), ref_idx)
    assert np.array_equal(cnt.cpu().numpy().reshape(-1), ref_cnt)
