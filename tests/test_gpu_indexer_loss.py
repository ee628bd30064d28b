"""GPU parity of the indexer auxiliary loss against the fp64 oracle.

Tolerances (max|err| <= tol * max|ref| per tensor), from the arithmetic:
* kl, dI: 1e-3. The kernel's logits are exact bf16 products summed in fp32 over
  Dqk terms, exponentiated with ex2.approx against the fp32 LSE; for N(0,1) inputs
  that bounds the exponent's error near 1e-4.
* dw: 1e-3 (exact z on dyadic inputs, fp32 sums).
* dq_idx, dk_idx: 2e-2. G = dI w [z > 0] is rounded to bf16 (2^-9 relative) before
  the tensor-core products, as dS and P are in the attention backward.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TOL, bf16_dev, dev, host_f64, rel_err
from synth import bf16_to_f32

pytestmark = pytest.mark.gpu

TOL_LOSS = 1e-3


def _dsa():
    import sparse_attention_index_gb300 as dsa
    return dsa


def _scores_dev(sc, B, S):
    """Oracle scores [B*S, S] (exact in fp32 on dyadic inputs) as a [B, S, ld] fp32 tensor."""
    ld = (S + 3) // 4 * 4
    a = np.full((B, S, ld), np.nan, dtype=np.float32)
    a[:, :, :S] = sc.reshape(B, S, S).astype(np.float32)
    return dev(a)


def _loss_case(B, S, H, Dqk, k, ndocs, seed, Hi=4, Di=32):
    Q = synth.normal_bf16((B, S, H, Dqk), seed, synth.STREAM_Q)
    K = synth.normal_bf16((B, S, 1, Dqk), seed, synth.STREAM_K)
    V = synth.normal_bf16((B, S, 1, 64), seed, synth.STREAM_V)
    q_idx = synth.dyadic_bf16((B, S, Hi, Di), seed, synth.STREAM_Q_IDX, -8, 8, 3)
    k_idx = synth.dyadic_bf16((B, S, Di), seed, synth.STREAM_K_IDX, -8, 8, 3)
    w = synth.dyadic_f32((B, S, Hi), seed, synth.STREAM_W, -1, 1, 4)
    seg = synth.segments(B, S, ndocs, seed) if ndocs else None
    sc = oracle.index_scores(q_idx, k_idx, w, seg)
    idx, _ = oracle.topk(sc, seg, S, k, B=B)
    idx = idx.reshape(B, S, k)
    scale = 1.0 / np.sqrt(Dqk)
    _, lse = oracle.attn_fwd(Q, K, V, idx, scale)
    return dict(Q=Q, K=K, q_idx=q_idx, k_idx=k_idx, w=w, sc=sc, idx=idx, lse=lse, scale=scale)


def _run_loss(c, B, S, g):
    dsa = _dsa()
    lse = dev(c["lse"].astype(np.float32).reshape(B, S, -1))
    kl, dI = dsa.dsa_indexer_loss(bf16_dev(c["Q"]), bf16_dev(c["K"]), dev(c["idx"]), lse,
                                  _scores_dev(c["sc"], B, S), c["scale"], g)
    assert dsa.dsa_get_last_device_error() == 0
    return host_f64(kl).reshape(-1), host_f64(dI).reshape(B * S, -1)


LOSS_CASES = [
    # B, S, H, Dqk, k, ndocs
    (1, 300, 128, 192, 64, 0),
    (2, 200, 16, 192, 100, 2),
    (1, 257, 5, 128, 300, 0),       # k > S: every causal key, a ragged last chunk
    (1, 129, 1, 192, 130, 0),
    (1, 500, 128, 128, 256, 3),     # two full chunks per late row
    (2, 150, 33, 192, 7, 0),        # H not a multiple of 16 or 32
    (1, 2300, 2, 128, 2200, 0),     # slots past the 16 chunks the kernel keeps from its pre-pass
]


@pytest.mark.parametrize("case", LOSS_CASES)
def test_indexer_loss_matches_oracle(case):
    B, S, H, Dqk, k, ndocs = case
    c = _loss_case(B, S, H, Dqk, k, ndocs, seed=700 + S + H)
    g = 0.5
    kl, dI = _run_loss(c, B, S, g)
    kl_ref, dI_ref = oracle.indexer_loss(c["Q"], c["K"], c["idx"], c["sc"], c["scale"], g)
    assert rel_err(kl, kl_ref) <= TOL_LOSS
    assert rel_err(dI, dI_ref) <= TOL_LOSS
    # slots without a selected key are exactly zero
    none = (c["idx"].reshape(B * S, k) < 0)
    assert np.all(dI[none] == 0.0)


def test_indexer_loss_user_lists_and_empty_rows():
    """-1 holes, keys above the diagonal, empty rows, unsorted lists, a duplicated key."""
    dsa = _dsa()
    B, S, H, Dqk, k = 1, 90, 16, 192, 70
    c = _loss_case(B, S, H, Dqk, 8, 0, seed=71)
    rng = np.random.default_rng(13)
    idx = np.full((B, S, k), -1, dtype=np.int32)
    for t in range(S):
        if t % 11 == 3:
            continue
        pick = rng.choice(S, size=min(S, k), replace=False).astype(np.int32)
        pick[rng.random(pick.size) < 0.2] = -1
        idx[0, t] = pick
    idx[0, 50, :3] = [7, 7, 20]                        # one key listed twice
    c["idx"] = idx
    V = synth.normal_bf16((B, S, 1, 64), 71, synth.STREAM_V)
    _, c["lse"] = oracle.attn_fwd(c["Q"], c["K"], V, idx, c["scale"])
    lse = c["lse"].astype(np.float32)
    lse[~np.isfinite(lse)] = 0.0                       # rows without keys: never read
    c["lse"] = lse
    kl, dI = _run_loss(c, B, S, 1.0)
    kl_ref, dI_ref = oracle.indexer_loss(c["Q"], c["K"], idx, c["sc"], c["scale"], 1.0)
    assert rel_err(kl, kl_ref) <= TOL_LOSS
    assert rel_err(dI, dI_ref) <= TOL_LOSS
    assert np.all(kl[3::11] == 0.0) and np.all(dI[3::11] == 0.0)


def _loss_bwd_case(B, S, k, ndocs, seed):
    c = _loss_case(B, S, 16, 192, k, ndocs, seed, Hi=64, Di=128)
    _, dI = oracle.indexer_loss(c["Q"], c["K"], c["idx"], c["sc"], c["scale"], 0.75)
    c["dI"] = dI.astype(np.float32)
    return c


LOSS_BWD_CASES = [
    # B, S, k, ndocs
    (1, 300, 64, 0),
    (2, 177, 61, 2),
    (1, 260, 300, 0),     # k > S
    (1, 400, 200, 3),
    (1, 129, 1, 0),       # one key per row
]


def _run_loss_bwd(c, B, S):
    dsa = _dsa()
    dq, dk, dw = dsa.dsa_indexer_loss_bwd(bf16_dev(c["q_idx"]), bf16_dev(c["k_idx"]), dev(c["w"]),
                                          dev(c["idx"]), dev(c["dI"].reshape(B, S, -1)))
    assert dsa.dsa_get_last_device_error() == 0
    return host_f64(dq), host_f64(dk), host_f64(dw)


@pytest.mark.parametrize("case", LOSS_BWD_CASES)
def test_indexer_loss_bwd_matches_oracle(case):
    B, S, k, ndocs = case
    c = _loss_bwd_case(B, S, k, ndocs, seed=800 + S)
    dq, dk, dw = _run_loss_bwd(c, B, S)
    dq_ref, dk_ref, dw_ref = oracle.indexer_loss_bwd(c["q_idx"], c["k_idx"], c["w"], c["idx"],
                                                     c["dI"].astype(np.float64))
    assert rel_err(dq.reshape(dq_ref.shape), dq_ref) <= TOL
    assert rel_err(dk, dk_ref) <= TOL
    assert rel_err(dw.reshape(dw_ref.shape), dw_ref) <= TOL_LOSS


def test_indexer_loss_chain_on_gpu_inputs():
    """scores, top-k and LSE from the library's own kernels, then the loss and its gradient,
    against the oracle run on the same (exact) scores and index lists."""
    dsa = _dsa()
    B, S, H, Dqk, k = 1, 384, 128, 192, 128
    seed = 91
    Q = synth.normal_bf16((B, S, H, Dqk), seed, synth.STREAM_Q)
    K = synth.normal_bf16((B, S, 1, Dqk), seed, synth.STREAM_K)
    V = synth.normal_bf16((B, S, 1, 128), seed, synth.STREAM_V)
    q_idx = synth.dyadic_bf16((B, S, 64, 128), seed, synth.STREAM_Q_IDX, -8, 8, 3)
    k_idx = synth.dyadic_bf16((B, S, 128), seed, synth.STREAM_K_IDX, -8, 8, 3)
    w = synth.dyadic_f32((B, S, 64), seed, synth.STREAM_W, -1, 1, 4)
    scale = Dqk ** -0.5
    qd, kd, wd = bf16_dev(q_idx), bf16_dev(k_idx), dev(w)
    Qd, Kd, Vd = bf16_dev(Q), bf16_dev(K), bf16_dev(V)
    scores = dsa.dsa_index_scores(qd, kd, wd)
    idx, _ = dsa.dsa_topk(scores, k)
    _, lse = dsa.dsa_sparse_attn_fwd(Qd, Kd, Vd, idx, scale)
    kl, dI = dsa.dsa_indexer_loss(Qd, Kd, idx, lse, scores, scale, 1.0)
    dq, dk, dw = dsa.dsa_indexer_loss_bwd(qd, kd, wd, idx, dI)
    assert dsa.dsa_get_last_device_error() == 0
    sc = oracle.index_scores(q_idx, k_idx, w, None)
    idx_ref, _ = oracle.topk(sc, None, S, k, B=B)
    assert np.array_equal(idx.cpu().numpy().reshape(-1, k), idx_ref)
    kl_ref, dI_ref = oracle.indexer_loss(Q, K, idx_ref.reshape(B, S, k), sc, scale, 1.0)
    assert rel_err(host_f64(kl).reshape(-1), kl_ref) <= TOL_LOSS
    assert rel_err(host_f64(dI).reshape(B * S, k), dI_ref) <= TOL_LOSS
    # the oracle's gradient from its own dI (the GPU's came from the GPU's dI)
    dq_ref, dk_ref, dw_ref = oracle.indexer_loss_bwd(q_idx, k_idx, w, idx_ref.reshape(B, S, k),
                                                     dI_ref)
    assert rel_err(host_f64(dq).reshape(dq_ref.shape), dq_ref) <= TOL
    assert rel_err(host_f64(dk), dk_ref) <= TOL
    assert rel_err(host_f64(dw).reshape(dw_ref.shape), dw_ref) <= TOL_LOSS


SIMT_LOSS_CASES = [
    # B, S, H, Hkv, Dqk, k: shapes the tensor-core kernel does not take
    (1, 128, 2, 1, 32, 4),        # the tiny workload's attention shape
    (1, 150, 8, 8, 64, 40),       # per-head K/V
    (2, 100, 6, 2, 48, 30),       # grouped heads, Dqk not a multiple of 64
]


def _simt_loss_case(B, S, H, Hkv, Dqk, k, seed):
    Q = synth.normal_bf16((B, S, H, Dqk), seed, synth.STREAM_Q)
    K = synth.normal_bf16((B, S, Hkv, Dqk), seed, synth.STREAM_K)
    V = synth.normal_bf16((B, S, Hkv, 32), seed, synth.STREAM_V)
    q_idx = synth.dyadic_bf16((B, S, 4, 32), seed, synth.STREAM_Q_IDX, -8, 8, 3)
    k_idx = synth.dyadic_bf16((B, S, 32), seed, synth.STREAM_K_IDX, -8, 8, 3)
    w = synth.dyadic_f32((B, S, 4), seed, synth.STREAM_W, -1, 1, 4)
    sc = oracle.index_scores(q_idx, k_idx, w, None)
    idx, _ = oracle.topk(sc, None, S, k, B=B)
    idx = idx.reshape(B, S, k)
    scale = 1.0 / np.sqrt(Dqk)
    _, lse = oracle.attn_fwd(Q, K, V, idx, scale)
    return dict(Q=Q, K=K, sc=sc, idx=idx, lse=lse, scale=scale)


@pytest.mark.parametrize("case", SIMT_LOSS_CASES)
def test_indexer_loss_cuda_core_shapes(case):
    """Shapes outside the tensor-core kernel (head dims, per-head or grouped K/V) run on the
    CUDA cores: same definition, same tolerances."""
    B, S, H, Hkv, Dqk, k = case
    c = _simt_loss_case(B, S, H, Hkv, Dqk, k, seed=930 + S + H)
    kl, dI = _run_loss(c, B, S, 0.5)
    kl_ref, dI_ref = oracle.indexer_loss(c["Q"], c["K"], c["idx"], c["sc"], c["scale"], 0.5)
    assert rel_err(kl, kl_ref) <= TOL_LOSS
    assert rel_err(dI, dI_ref) <= TOL_LOSS


@pytest.mark.parametrize("Hi, Di", [(4, 32), (32, 64), (16, 128)])
def test_indexer_loss_bwd_cuda_core_shapes(Hi, Di):
    """Index shapes other than 64 x 128 run on the CUDA cores in fp32 (no bf16 rounding of G)."""
    dsa = _dsa()
    B, S, k = 1, 160, 48
    seed = 940 + Hi + Di
    q_idx = synth.dyadic_bf16((B, S, Hi, Di), seed, synth.STREAM_Q_IDX, -8, 8, 3)
    k_idx = synth.dyadic_bf16((B, S, Di), seed, synth.STREAM_K_IDX, -8, 8, 3)
    w = synth.dyadic_f32((B, S, Hi), seed, synth.STREAM_W, -1, 1, 4)
    sc = oracle.index_scores(q_idx, k_idx, w, None)
    idx, _ = oracle.topk(sc, None, S, k, B=B)
    idx = idx.reshape(B, S, k)
    dI = synth.normal_bf16((B * S, k), seed, synth.STREAM_DO)
    dI = np.where(idx.reshape(B * S, k) >= 0, bf16_to_f32(dI), 0.0).astype(np.float32)
    dq, dk, dw = dsa.dsa_indexer_loss_bwd(bf16_dev(q_idx), bf16_dev(k_idx), dev(w), dev(idx),
                                          dev(dI.reshape(B, S, k)))
    assert dsa.dsa_get_last_device_error() == 0
    dq_ref, dk_ref, dw_ref = oracle.indexer_loss_bwd(q_idx, k_idx, w, idx, dI.astype(np.float64))
    assert rel_err(host_f64(dq).reshape(dq_ref.shape), dq_ref) <= TOL_LOSS
    assert rel_err(host_f64(dk), dk_ref) <= TOL_LOSS
    assert rel_err(host_f64(dw).reshape(dw_ref.shape), dw_ref) <= TOL_LOSS


def test_indexer_loss_refusals():
    dsa = _dsa()
    B, S, k = 1, 64, 16
    idx = torch.full((B, S, k), -1, dtype=torch.int32, device="cuda")
    lse = torch.zeros((B, S, 6), device="cuda")
    sc = torch.zeros((B, S, S), device="cuda")
    Q = torch.zeros((B, S, 6, 64), dtype=torch.bfloat16, device="cuda")
    K = torch.zeros((B, S, 4, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dsa.DsaError) as e:
        dsa.dsa_indexer_loss(Q, K, idx, lse, sc, 0.1)        # 4 K/V heads do not divide 6
    assert e.value.status == dsa.DSA_ERR_INVALID_ARG
    qi = torch.zeros((B, S, 128, 512), dtype=torch.bfloat16, device="cuda")
    ki = torch.zeros((B, S, 512), dtype=torch.bfloat16, device="cuda")
    wi = torch.zeros((B, S, 128), device="cuda")
    dI = torch.zeros((B, S, k), device="cuda")
    with pytest.raises(dsa.DsaError) as e:
        dsa.dsa_indexer_loss_bwd(qi, ki, wi, idx, dI)          # Hi * (Di + 1) > 51200
    assert e.value.status == dsa.DSA_ERR_UNSUPPORTED
    assert dsa.dsa_get_last_device_error() == 0


def test_indexer_loss_bad_index_is_reported():
    dsa = _dsa()
    B, S, H, Dqk, k = 1, 100, 16, 128, 20
    c = _loss_case(B, S, H, Dqk, k, 0, seed=17)
    idx = c["idx"].copy()
    idx[0, 60, 3] = S + 5                               # out of range: skipped and reported
    lse = dev(c["lse"].astype(np.float32).reshape(B, S, -1))
    dsa.dsa_indexer_loss(bf16_dev(c["Q"]), bf16_dev(c["K"]), dev(idx), lse,
                         _scores_dev(c["sc"], B, S), c["scale"], 1.0)
    code = dsa.dsa_get_last_device_error()
    assert code == (dsa.DSA_STAGE_LOSS | dsa.DSA_DEVERR_BAD_INDEX)
