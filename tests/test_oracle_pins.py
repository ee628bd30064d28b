"""Pins for the fp64 oracle: each check rests on something other than the oracle itself.

* indexer - special cases that reduce to a matrix product (numpy), the identity
  ReLU(x) - ReLU(-x) = x, exactness on dyadic inputs, mask structure;
* top-k - hand-derived fixtures (tests/golden/topk_ties.txt), exhaustive subset
  search on tiny rows, numpy lexsort, invariants;
* attention - dense masked attention through torch's scaled_dot_product_attention
  in fp64 (index mask built from the selected lists), closed forms (first token,
  constant keys), permutation invariance;
* backward - torch.autograd in fp64 through the same dense routine, central
  finite differences of the oracle forward, and closed-form sums.
"""
import itertools
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import bf16_bits_to_f64, f64_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- fixtures

def _dyadic_inputs(B, S, Hi, Di, seed, lo=-8, hi=8, nonneg=False, seg_docs=0):
    if nonneg:
        lo = 0
    q = synth.dyadic_bf16((B, S, Hi, Di), seed, 1, lo, hi, 3)
    k = synth.dyadic_bf16((B, S, Di), seed, 2, lo, hi, 3)
    w = synth.dyadic_f32((B, S, Hi), seed, 3, 0 if nonneg else -4, 4, 4)
    seg = synth.segments(B, S, seg_docs, seed) if seg_docs else None
    return q, k, w, seg


def _negate_bf16(u16):
    return (u16 ^ np.uint16(0x8000)).astype(np.uint16)


# ------------------------------------------------------------------ indexer

def test_indexer_single_head_unit_weight_is_relu_of_matmul():
    """Hi = 1, w = 1: I[t, s] = ReLU(q[t] . k[s]) - one matrix product."""
    B, S, Di = 2, 37, 24
    q, k, _, _ = _dyadic_inputs(B, S, 1, Di, seed=11)
    w = np.ones((B, S, 1), dtype=np.float32)
    got = oracle.index_scores(q, k, w, None)
    qf, kf = bf16_bits_to_f64(q)[:, :, 0, :], bf16_bits_to_f64(k)
    for b in range(B):
        ref = np.maximum(qf[b] @ kf[b].T, 0.0)
        for t in range(S):
            np.testing.assert_array_equal(got[b * S + t, : t + 1], ref[t, : t + 1])


def test_indexer_nonnegative_inputs_collapse_heads():
    """q, k, w >= 0 make every ReLU the identity, so I[t,:] = (w[t] @ q[t]) @ k^T."""
    B, S, Hi, Di = 2, 29, 5, 16
    q, k, w, _ = _dyadic_inputs(B, S, Hi, Di, seed=12, nonneg=True)
    got = oracle.index_scores(q, k, w, None)
    qf, kf = bf16_bits_to_f64(q), bf16_bits_to_f64(k)
    for b in range(B):
        for t in range(S):
            wq = w[b, t].astype(np.float64) @ qf[b, t]          # [Di]
            ref = kf[b, : t + 1] @ wq
            np.testing.assert_array_equal(got[b * S + t, : t + 1], ref)


def test_indexer_relu_split_identity():
    """ReLU(x) - ReLU(-x) = x: I(q, k) - I(q, -k) = sum_h w[t,h] q[t,h] . k[s] for any signs."""
    B, S, Hi, Di = 1, 41, 7, 32
    q, k, w, _ = _dyadic_inputs(B, S, Hi, Di, seed=13)
    plus = oracle.index_scores(q, k, w, None)
    minus = oracle.index_scores(q, _negate_bf16(k), w, None)
    qf, kf = bf16_bits_to_f64(q), bf16_bits_to_f64(k)
    for t in range(S):
        wq = w[0, t].astype(np.float64) @ qf[0, t]
        np.testing.assert_array_equal(plus[t, : t + 1] - minus[t, : t + 1], kf[0, : t + 1] @ wq)
    # all dot products <= 0  =>  every score is exactly zero
    qn, kn, wn, _ = _dyadic_inputs(B, S, Hi, Di, seed=14, nonneg=True)
    zero = oracle.index_scores(qn, _negate_bf16(kn), w, None)
    for t in range(S):
        assert np.all(zero[t, : t + 1] == 0.0)


def test_indexer_mask_structure_and_segments():
    """NaN above the diagonal; -inf exactly where the document differs; finite elsewhere."""
    B, S, Hi, Di = 2, 53, 4, 16
    q, k, w, seg = _dyadic_inputs(B, S, Hi, Di, seed=15, seg_docs=3)
    got = oracle.index_scores(q, k, w, seg)
    plain = oracle.index_scores(q, k, w, None)
    for b in range(B):
        for t in range(S):
            row = got[b * S + t]
            assert np.all(np.isnan(row[t + 1:]))
            same = seg[b, : t + 1] == seg[b, t]
            assert np.all(np.isneginf(row[: t + 1][~same]))
            np.testing.assert_array_equal(row[: t + 1][same], plain[b * S + t, : t + 1][same])
            assert same[t]


def test_indexer_dyadic_workload_is_exact_in_fp32():
    """On the dyadic workloads every score is an fp32 value (the GPU must match bit for bit)."""
    wl = synth.WORKLOADS["packed_s489"]
    inp = synth.indexer_inputs(wl)
    rows = synth.sample_rows(wl, 24)
    got = oracle.index_scores(inp["q_idx"], inp["k_idx"], inp["w"], inp["seg"], rows=rows)
    finite = np.isfinite(got)
    assert np.all(got[finite].astype(np.float32).astype(np.float64) == got[finite])
    # granularity 2^-10 (q, k in 1/8 steps, w in 1/16 steps)
    assert np.all(np.mod(got[finite] * 1024.0, 1.0) == 0.0)


def test_indexer_weight_homogeneity_and_linearity():
    """I is linear in w: I(2 w) = 2 I(w); I(w1 + w2) = I(w1) + I(w2)."""
    B, S, Hi, Di = 1, 23, 6, 16
    q, k, w, _ = _dyadic_inputs(B, S, Hi, Di, seed=16)
    w2 = synth.dyadic_f32((B, S, Hi), 99, 3, -4, 4, 4)
    a = oracle.index_scores(q, k, w, None)
    b2 = oracle.index_scores(q, k, w2, None)
    ab = oracle.index_scores(q, k, (w + w2).astype(np.float32), None)
    d = oracle.index_scores(q, k, (2 * w).astype(np.float32), None)
    for t in range(S):
        np.testing.assert_array_equal(d[t, : t + 1], 2 * a[t, : t + 1])
        np.testing.assert_array_equal(ab[t, : t + 1], a[t, : t + 1] + b2[t, : t + 1])


def test_indexer_integer_inputs_match_exact_int64_arithmetic():
    """Integer q, k and w: every score is an integer, computed here in numpy int64 with
    no floating point at all (per head, per key: a dot product, a max with 0, a weight)."""
    B, S, Hi, Di = 2, 45, 5, 24
    q = synth.dyadic_bf16((B, S, Hi, Di), 41, 1, -4, 4, 0)
    k = synth.dyadic_bf16((B, S, Di), 41, 2, -4, 4, 0)
    w = synth.dyadic_f32((B, S, Hi), 41, 3, -3, 3, 0)
    got = oracle.index_scores(q, k, w, None)
    qi = bf16_bits_to_f64(q).astype(np.int64)
    ki = bf16_bits_to_f64(k).astype(np.int64)
    wi = w.astype(np.int64)
    assert np.array_equal(qi, bf16_bits_to_f64(q)) and np.array_equal(wi, w)
    for b in range(B):
        z = np.einsum("thd,sd->ths", qi[b], ki[b])                 # int64 [S, Hi, S]
        ref = np.einsum("th,ths->ts", wi[b], np.maximum(z, 0))     # int64 [S, S]
        for t in range(S):
            np.testing.assert_array_equal(got[b * S + t, : t + 1], ref[t, : t + 1])


def test_indexer_matches_fp64_torch_matmul_of_the_dense_product():
    """One fp64 torch.matmul of [S*Hi, Di] x [Di, S], then ReLU, the head weights and the
    sum over heads: the scores of every causal pair, on the dyadic tiny workload."""
    wl = synth.WORKLOADS["tiny_s128"]
    inp = synth.indexer_inputs(wl)
    got = oracle.index_scores(inp["q_idx"], inp["k_idx"], inp["w"], None)
    S, Hi, Di = wl.S, wl.Hi, wl.Di
    q = torch.from_numpy(bf16_bits_to_f64(inp["q_idx"])[0].reshape(S * Hi, Di))
    k = torch.from_numpy(bf16_bits_to_f64(inp["k_idx"])[0])
    z = torch.matmul(q, k.T).reshape(S, Hi, S)
    w = torch.from_numpy(inp["w"][0].astype(np.float64))
    ref = (w[:, :, None] * torch.relu(z)).sum(1).numpy()
    tri = np.tril(np.ones((S, S), dtype=bool))
    np.testing.assert_array_equal(got[:, :S][tri], ref[tri])


# ------------------------------------------------------- fp8 index scores

# OCP 8-bit floating point specification, E4M3 (bias 7, exponent 0 subnormal,
# S.1111.111 NaN, no infinities): byte -> value
E4M3_SPEC = [(0x00, 0.0), (0x80, -0.0), (0x38, 1.0), (0xB8, -1.0), (0x30, 0.5), (0x3C, 1.5),
             (0x40, 2.0), (0x44, 3.0), (0x7E, 448.0), (0xFE, -448.0), (0x08, 2.0 ** -6),
             (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x77, 240.0), (0x28, 0.25), (0x20, 0.125)]


def test_e4m3_decode_spec_values():
    got = oracle.e4m3_decode(np.array([b for b, _ in E4M3_SPEC], dtype=np.uint8))
    for (b, v), g in zip(E4M3_SPEC, got):
        assert g == v and np.signbit(g) == np.signbit(v), (hex(b), g, v)
    nan = oracle.e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))
    assert np.all(np.isnan(nan))


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.signbit(got[fin]), np.signbit(ref[fin]))


def _fp8_case(B, S, Hi, Di, seed, k_scale):
    wl = synth.Workload("fp8pin", seed=seed, B=B, S=S, Hi=Hi, Di=Di, topk=4, H=1, Dqk=32, Dv=32,
                        backward=False)
    return synth.indexer_inputs_fp8(wl, k_scale)


def test_indexer_fp8_brute_force_tiny():
    """Against a numpy einsum on torch-decoded inputs, scale applied to k."""
    B, S, Hi, Di = 1, 9, 3, 8
    inp = _fp8_case(B, S, Hi, Di, seed=31, k_scale="dyadic")
    dec = lambda a: torch.from_numpy(a).view(torch.float8_e4m3fn).to(torch.float64).numpy()  # noqa: E731
    q, k = dec(inp["q_idx"])[0], dec(inp["k_idx"])[0] * inp["k_scale"][0][:, None]
    dots = np.einsum("thd,sd->tsh", q, k)
    ref = np.einsum("tsh,th->ts", np.maximum(dots, 0.0), inp["w"][0].astype(np.float64))
    got = oracle.index_scores_fp8(inp["q_idx"], inp["k_idx"], inp["w"], None, inp["k_scale"])
    for t in range(S):
        np.testing.assert_allclose(got[t, : t + 1], ref[t, : t + 1], rtol=1e-14, atol=0)
        assert np.all(np.isnan(got[t, t + 1:]))


def test_indexer_fp8_equals_bf16_definition_on_same_values():
    wl = synth.WORKLOADS["packed_s489"]
    rows = synth.sample_rows(wl, 12)
    a = synth.indexer_inputs(wl)
    f = synth.indexer_inputs_fp8(wl, "none")
    ref = oracle.index_scores(a["q_idx"], a["k_idx"], a["w"], a["seg"], rows=rows)
    got = oracle.index_scores_fp8(f["q_idx"], f["k_idx"], f["w"], f["seg"], rows=rows)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])


def test_indexer_fp8_positive_key_scale_is_homogeneous():
    """relu(q . c k) = c relu(q . k) for c > 0: a power-of-two scale multiplies each score."""
    B, S, Hi, Di = 2, 40, 4, 16
    f = _fp8_case(B, S, Hi, Di, seed=32, k_scale="pow2")
    plain = oracle.index_scores_fp8(f["q_idx"], f["k_idx"], f["w"], None)
    scaled = oracle.index_scores_fp8(f["q_idx"], f["k_idx"], f["w"], None, f["k_scale"])
    for b in range(B):
        for t in range(S):
            r = b * S + t
            np.testing.assert_array_equal(scaled[r, : t + 1],
                                          plain[r, : t + 1] * f["k_scale"][b, : t + 1])


# ------------------------------------------------------------------- top-k

def _parse_golden():
    cases = []
    with open(os.path.join(GOLDEN, "topk_ties.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, seg, scores, expect = [p.strip() for p in line.split("|")]
            cases.append((int(k), None if seg == "-" else [int(x) for x in seg.split()],
                          [float(x) for x in scores.split()], [int(x) for x in expect.split()]))
    return cases


@pytest.mark.parametrize("case", _parse_golden())
def test_topk_golden_fixtures(case):
    k, seg, scores, expect = case
    S = len(scores)
    t = S - 1
    sc = np.full((1, S), np.nan)
    sc[0, : t + 1] = scores
    seg_a = None if seg is None else np.array([seg], dtype=np.int32)
    idx, cnt = oracle.topk(sc, seg_a, S, k, rows=np.array([t]))
    assert idx[0].tolist() == expect
    assert cnt[0] == sum(1 for x in expect if x >= 0)


def _brute_force_topk(scores, valid, k):
    """The unique subset T, |T| = min(k, n), such that every s in T beats every u not in T."""
    cand = [s for s in range(len(scores)) if valid[s]]
    m = min(k, len(cand))

    def beats(s, u):
        return scores[s] > scores[u] or (scores[s] == scores[u] and s < u)

    found = []
    for T in itertools.combinations(cand, m):
        rest = [u for u in cand if u not in T]
        if all(beats(s, u) for s in T for u in rest):
            found.append(list(T))
    assert len(found) == 1
    return found[0] + [-1] * (k - m)


def test_topk_exhaustive_subset_search_tiny_rows():
    rng = np.random.default_rng(5)
    S = 9
    for trial in range(60):
        k = int(rng.integers(1, 6))
        vals = rng.choice([-1.0, -0.0, 0.0, 0.5, 0.5, 2.0], size=S)   # many ties, both zeros
        seg = np.sort(rng.integers(0, 3, size=S)).astype(np.int32)[None] if trial % 2 else None
        sc = np.tile(vals, (S, 1))
        rows = np.arange(S)
        idx, _ = oracle.topk(sc, seg, S, k, rows=rows)
        for t in range(S):
            valid = [s <= t and (seg is None or seg[0, s] == seg[0, t]) for s in range(S)]
            assert idx[t].tolist() == _brute_force_topk(list(vals), valid, k)


def test_topk_matches_numpy_lexsort():
    """Library route: np.lexsort on (s, -score) gives the same selection."""
    wl = synth.WORKLOADS["tiny_s128"]
    inp = synth.indexer_inputs(wl)
    sc = oracle.index_scores(inp["q_idx"], inp["k_idx"], inp["w"], None)
    idx, cnt = oracle.topk(sc, None, wl.S, wl.topk)
    for t in range(wl.S):
        s_idx = np.arange(t + 1)
        order = np.lexsort((s_idx, -sc[t, : t + 1]))
        m = min(wl.topk, t + 1)
        exp = np.sort(order[:m]).tolist() + [-1] * (wl.topk - m)
        assert idx[t].tolist() == exp
        assert cnt[t] == m


@pytest.mark.parametrize("name", ["tiny_s128", "packed_s489"])
def test_topk_invariants_on_workloads(name):
    wl = synth.WORKLOADS[name]
    inp = synth.indexer_inputs(wl)
    rows = synth.sample_rows(wl, 40)
    sc = oracle.index_scores(inp["q_idx"], inp["k_idx"], inp["w"], inp["seg"], rows=rows)
    idx, cnt = oracle.topk(sc, inp["seg"], wl.S, wl.topk, rows=rows, B=wl.B)
    seg = inp["seg"]
    for r, row in enumerate(rows):
        b, t = divmod(int(row), wl.S)
        valid = np.array([seg is None or seg[b, s] == seg[b, t] for s in range(t + 1)])
        n = int(valid.sum())
        m = min(wl.topk, n)
        sel = idx[r, :m]
        assert cnt[r] == m
        assert np.all(idx[r, m:] == -1)
        assert np.all(np.diff(sel) > 0)
        assert np.all(sel <= t) and np.all(valid[sel])
        chosen = np.zeros(t + 1, bool)
        chosen[sel] = True
        rest = valid & ~chosen
        if rest.any():
            lo = sc[r, : t + 1][chosen].min()
            hi = sc[r, : t + 1][rest].max()
            assert lo >= hi
            # ties at the threshold went to the lower indices
            tie_sel = np.nonzero(chosen & (sc[r, : t + 1] == lo))[0]
            tie_rest = np.nonzero(rest & (sc[r, : t + 1] == lo))[0]
            if tie_rest.size:
                assert tie_sel.max() < tie_rest.min()
        if wl.topk >= n:
            assert chosen[valid].all()


# --------------------------------------------------------------- attention

def _attn_case(B, S, H, Hkv, Dqk, Dv, seed, k, seg_docs=0):
    Q = synth.normal_bf16((B, S, H, Dqk), seed, 4)
    K = synth.normal_bf16((B, S, Hkv, Dqk), seed, 5)
    V = synth.normal_bf16((B, S, Hkv, Dv), seed, 6)
    dO = synth.normal_bf16((B, S, H, Dv), seed, 7)
    seg = synth.segments(B, S, seg_docs, seed) if seg_docs else None
    # a selection from the oracle's own top-k over oracle index scores
    Hi, Di = 3, 16
    q_idx = synth.dyadic_bf16((B, S, Hi, Di), seed, 1, -8, 8, 3)
    k_idx = synth.dyadic_bf16((B, S, Di), seed, 2, -8, 8, 3)
    w = synth.dyadic_f32((B, S, Hi), seed, 3, -4, 4, 4)
    sc = oracle.index_scores(q_idx, k_idx, w, seg)
    idx, _ = oracle.topk(sc, seg, S, k, B=B)
    return Q, K, V, dO, idx.reshape(B, S, k), seg


def _dense_mask(idx, S):
    """Boolean [B, S, S] mask: causal AND selected (the index mask of the pages)."""
    B, _, k = idx.shape
    m = np.zeros((B, S, S), dtype=bool)
    for b in range(B):
        for t in range(S):
            for s in idx[b, t]:
                if 0 <= s <= t:
                    m[b, t, s] = True
    return m


def _torch_dense(Q, K, V, mask, scale, H, Hkv, requires_grad=False):
    q = torch.from_numpy(bf16_bits_to_f64(Q)).permute(0, 2, 1, 3).contiguous()
    k = torch.from_numpy(bf16_bits_to_f64(K)).permute(0, 2, 1, 3).contiguous()
    v = torch.from_numpy(bf16_bits_to_f64(V)).permute(0, 2, 1, 3).contiguous()
    for x in (q, k, v):
        x.requires_grad_(requires_grad)
    kk = k.repeat_interleave(H // Hkv, dim=1)
    vv = v.repeat_interleave(H // Hkv, dim=1)
    am = torch.from_numpy(mask)[:, None, :, :]
    o = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, attn_mask=am, scale=scale)
    return q, k, v, o


@pytest.mark.parametrize("Hkv", [1, 4])
@pytest.mark.parametrize("seg_docs", [0, 3])
def test_attn_fwd_matches_dense_sdpa(Hkv, seg_docs):
    B, S, H, Dqk, Dv, k = 2, 40, 4, 24, 16, 7
    Q, K, V, _, idx, seg = _attn_case(B, S, H, Hkv, Dqk, Dv, seed=21, k=k, seg_docs=seg_docs)
    scale = 1 / np.sqrt(Dqk)
    O, lse = oracle.attn_fwd(Q, K, V, idx, scale)
    _, _, _, o = _torch_dense(Q, K, V, _dense_mask(idx, S), scale, H, Hkv)
    ref = o.permute(0, 2, 1, 3).reshape(B * S, H, Dv).numpy()
    np.testing.assert_allclose(O, ref, rtol=1e-12, atol=1e-12)
    # LSE: softmax weights recovered from it sum to one (closed form of log-sum-exp)
    assert np.all(np.isfinite(lse))


def test_attn_fwd_k_at_least_s_is_dense_causal_attention():
    """k >= S selects every causal key: the result is plain causal softmax attention."""
    B, S, H, Dqk, Dv = 1, 33, 3, 16, 8
    Q, K, V, _, idx, _ = _attn_case(B, S, H, 1, Dqk, Dv, seed=22, k=S + 3)
    assert np.all((idx[0] >= 0).sum(-1) == np.arange(1, S + 1))
    scale = 0.37
    O, lse = oracle.attn_fwd(Q, K, V, idx, scale)
    q = torch.from_numpy(bf16_bits_to_f64(Q)).permute(0, 2, 1, 3)
    k = torch.from_numpy(bf16_bits_to_f64(K)).permute(0, 2, 1, 3).expand(B, H, S, Dqk)
    v = torch.from_numpy(bf16_bits_to_f64(V)).permute(0, 2, 1, 3).expand(B, H, S, Dv)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=scale)
    np.testing.assert_allclose(O, o.permute(0, 2, 1, 3).reshape(S, H, Dv).numpy(), rtol=1e-12,
                               atol=1e-12)
    logits = torch.einsum("bhtd,bhsd->bhts", q, k) * scale
    logits = logits.masked_fill(~torch.ones(S, S, dtype=torch.bool).tril(), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(logits, -1)[0].T.numpy(), rtol=1e-12)


def test_attn_fwd_closed_forms():
    B, S, H, Dqk, Dv, k = 1, 20, 2, 16, 8, 5
    Q, K, V, _, idx, _ = _attn_case(B, S, H, 1, Dqk, Dv, seed=23, k=k)
    scale = 0.25
    O, lse = oracle.attn_fwd(Q, K, V, idx, scale)
    Vf, Qf, Kf = bf16_bits_to_f64(V), bf16_bits_to_f64(Q), bf16_bits_to_f64(K)
    # first token: one key, so O = V[0] and LSE = scale * q . k
    np.testing.assert_array_equal(O[0], np.tile(Vf[0, 0, 0], (H, 1)))
    np.testing.assert_allclose(lse[0], scale * Qf[0, 0] @ Kf[0, 0, 0], rtol=1e-14)
    # all-zero keys: uniform weights, O = mean of the selected values, LSE = log m
    Kz = np.zeros_like(K)
    Oz, lz = oracle.attn_fwd(Q, Kz, V, idx, scale)
    for t in range(S):
        sel = idx[0, t][idx[0, t] >= 0]
        np.testing.assert_allclose(Oz[t], np.tile(Vf[0, sel, 0].mean(0), (H, 1)), rtol=1e-13)
        np.testing.assert_allclose(lz[t], np.log(len(sel)), rtol=1e-14)
    # order of the selected list does not matter (it is a mask)
    perm = idx.copy()
    rng = np.random.default_rng(0)
    for t in range(S):
        rng.shuffle(perm[0, t])
    Op, lp = oracle.attn_fwd(Q, K, V, perm, scale)
    np.testing.assert_allclose(Op, O, rtol=1e-13, atol=1e-15)
    # keys above the diagonal in the list are masked out by causality
    bad = idx.copy()
    bad[0, 3, -1] = 10
    Ob, _ = oracle.attn_fwd(Q, K, V, bad, scale)
    np.testing.assert_array_equal(Ob[3], O[3])


def test_attn_empty_selection():
    B, S, H, D = 1, 4, 2, 16
    Q = synth.normal_bf16((B, S, H, D), 1, 4)
    K = synth.normal_bf16((B, S, 1, D), 1, 5)
    V = synth.normal_bf16((B, S, 1, D), 1, 6)
    idx = np.full((B, S, 3), -1, dtype=np.int32)
    O, lse = oracle.attn_fwd(Q, K, V, idx, 0.25)
    assert np.all(O == 0) and np.all(np.isneginf(lse))


# ----------------------------------------------------------------- backward

@pytest.mark.parametrize("Hkv", [1, 2])
@pytest.mark.parametrize("seg_docs", [0, 3])
def test_attn_bwd_matches_torch_autograd(Hkv, seg_docs):
    B, S, H, Dqk, Dv, k = 2, 30, 4, 16, 8, 6
    Q, K, V, dO, idx, seg = _attn_case(B, S, H, Hkv, Dqk, Dv, seed=31, k=k, seg_docs=seg_docs)
    scale = 1 / np.sqrt(Dqk)
    dQ, dK, dV = oracle.attn_bwd(Q, K, V, idx, dO, scale)
    q, kt, vt, o = _torch_dense(Q, K, V, _dense_mask(idx, S), scale, H, Hkv, requires_grad=True)
    g = torch.from_numpy(bf16_bits_to_f64(dO)).permute(0, 2, 1, 3)
    (o * g).sum().backward()
    np.testing.assert_allclose(dQ, q.grad.permute(0, 2, 1, 3).reshape(B * S, H, Dqk).numpy(),
                               rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dK, kt.grad.permute(0, 2, 1, 3).numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dV, vt.grad.permute(0, 2, 1, 3).numpy(), rtol=1e-10, atol=1e-12)


def test_attn_bwd_finite_differences():
    """Central differences of L = <dO, O> with a step of 2^-6 on exactly representable entries."""
    B, S, H, Dqk, Dv, k = 1, 12, 2, 16, 8, 4
    Q, K, V, dO, idx, _ = _attn_case(B, S, H, 1, Dqk, Dv, seed=32, k=k)
    # move the probed entries to 1.0 so that 1 +- 2^-6 are bf16 values
    probes = [("Q", (0, 9, 1, 3)), ("Q", (0, 4, 0, 0)), ("K", (0, 2, 0, 5)), ("K", (0, 7, 0, 1)),
              ("V", (0, 3, 0, 2)), ("V", (0, 8, 0, 7))]
    arrs = {"Q": Q.copy(), "K": K.copy(), "V": V.copy()}
    for name, ix in probes:
        arrs[name][ix] = f64_to_bf16_bits(np.array([1.0]))[0]
    scale = 0.3
    dQ, dK, dV = oracle.attn_bwd(arrs["Q"], arrs["K"], arrs["V"], idx, dO, scale)
    grads = {"Q": dQ.reshape(B, S, H, Dqk), "K": dK, "V": dV}
    dOf = bf16_bits_to_f64(dO).reshape(B * S, H, Dv)
    eps = 2.0 ** -6

    def loss(a):
        O, _ = oracle.attn_fwd(a["Q"], a["K"], a["V"], idx, scale)
        return float((O * dOf).sum())

    for name, ix in probes:
        vals = []
        for sgn in (+1, -1):
            a = {n: x.copy() for n, x in arrs.items()}
            a[name][ix] = f64_to_bf16_bits(np.array([1.0 + sgn * eps]))[0]
            vals.append(loss(a))
        fd = (vals[0] - vals[1]) / (2 * eps)
        an = grads[name][ix]
        assert abs(fd - an) <= 2e-3 * max(1.0, abs(an)), (name, ix, fd, an)


def test_attn_bwd_closed_form_sums():
    B, S, H, Dqk, Dv, k = 2, 25, 3, 16, 8, 5
    Q, K, V, dO, idx, _ = _attn_case(B, S, H, 1, Dqk, Dv, seed=33, k=k)
    scale = 0.2
    dQ, dK, dV = oracle.attn_bwd(Q, K, V, idx, dO, scale)
    # softmax weights sum to one: sum over keys of dV equals sum over queries and heads of dO
    dOf = bf16_bits_to_f64(dO)
    np.testing.assert_allclose(dV.sum(axis=(1, 2)), dOf.sum(axis=(1, 2)), rtol=1e-12, atol=1e-12)
    # the rows of dS sum to zero: with every key equal to one vector c, dQ = 0
    Kc = np.tile(K[:, :1], (1, S, 1, 1))
    dQc, dKc, _ = oracle.attn_bwd(Q, Kc, V, idx, dO, scale)
    assert np.max(np.abs(dQc)) < 1e-12
    # ... and dK summed over keys is zero as well (sum_j dS_j = 0 for every query)
    np.testing.assert_allclose(dK.sum(axis=1), 0.0, atol=1e-11)
    # a subset of rows contributes a part: partial sums over a row split add up
    rows_a = np.arange(0, B * S, 2)
    rows_b = np.arange(1, B * S, 2)
    _, dKa, dVa = oracle.attn_bwd(Q, K, V, idx, dO, scale, rows=rows_a)
    _, dKb, dVb = oracle.attn_bwd(Q, K, V, idx, dO, scale, rows=rows_b)
    np.testing.assert_allclose(dKa + dKb, dK, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dVa + dVb, dV, rtol=1e-12, atol=1e-13)


def test_attn_bwd_unselected_keys_get_no_gradient():
    """A key that no query lists receives no gradient: dK = dV = 0 there, exactly. The
    selection keeps only even keys, and key S - 1 (odd) is listed by nobody else either."""
    B, S, H, Dqk, Dv = 1, 24, 3, 16, 8
    Q, K, V, dO, _, _ = _attn_case(B, S, H, 1, Dqk, Dv, seed=34, k=4)
    idx = np.full((B, S, 6), -1, dtype=np.int32)
    for t in range(S):
        evens = [s for s in range(0, t + 1, 2)][-6:]
        idx[0, t, : len(evens)] = evens
    dQ, dK, dV = oracle.attn_bwd(Q, K, V, idx, dO, 0.25)
    odd = np.arange(1, S, 2)
    assert np.all(dK[0, odd] == 0.0) and np.all(dV[0, odd] == 0.0)
    # the listed keys do get some gradient (the test is not vacuous)
    listed = np.unique(idx[idx >= 0])
    assert np.all(np.abs(dV[0, listed]).sum(-1).sum(-1) > 0)


# ------------------------------------------------------------- indexer loss

def _iloss_case(B, S, H, Dqk, seed, k, Hi=3, Di=16, seg_docs=0):
    Q = synth.normal_bf16((B, S, H, Dqk), seed, 4)
    K = synth.normal_bf16((B, S, 1, Dqk), seed, 5)
    seg = synth.segments(B, S, seg_docs, seed) if seg_docs else None
    q_idx = synth.dyadic_bf16((B, S, Hi, Di), seed, 1, -8, 8, 3)
    k_idx = synth.dyadic_bf16((B, S, Di), seed, 2, -8, 8, 3)
    w = synth.dyadic_f32((B, S, Hi), seed, 3, -4, 4, 4)
    sc = oracle.index_scores(q_idx, k_idx, w, seg)
    idx, _ = oracle.topk(sc, seg, S, k, B=B)
    return Q, K, q_idx, k_idx, w, seg, sc, idx.reshape(B, S, k)


def _torch_teacher_student(Q, K, idx, scores, scale, H):
    """Dense fp64 torch: target pbar [B,S,S] and log-student [B,S,S] under the index mask."""
    B, S = Q.shape[:2]
    mask = torch.from_numpy(_dense_mask(idx, S))
    q = torch.from_numpy(bf16_bits_to_f64(Q))                       # [B,S,H,D]
    kk = torch.from_numpy(bf16_bits_to_f64(K))[:, :, 0]              # [B,S,D]
    logits = torch.einsum("bthd,bsd->bhts", q, kk) * scale
    logits = logits.masked_fill(~mask[:, None], float("-inf"))
    probs = torch.softmax(logits, dim=-1)
    probs = torch.nan_to_num(probs, nan=0.0)                         # rows without a key
    pbar = probs.sum(dim=1) / H
    I = torch.from_numpy(np.nan_to_num(scores.reshape(B, S, S), nan=-np.inf))
    return pbar, I, mask


def _slots_to_dense(vals, idx, S):
    B, _, k = idx.shape
    out = np.zeros((B, S, S))
    v = vals.reshape(B, S, k)
    for b in range(B):
        for t in range(S):
            for j in range(k):
                s = idx[b, t, j]
                if 0 <= s <= t:
                    out[b, t, s] += v[b, t, j]
    return out


@pytest.mark.parametrize("seg_docs", [0, 3])
def test_indexer_loss_matches_torch_kl_div_and_autograd(seg_docs):
    B, S, H, Dqk, k = 2, 36, 5, 24, 6
    Q, K, _, _, _, seg, sc, idx = _iloss_case(B, S, H, Dqk, seed=41, k=k, seg_docs=seg_docs)
    scale, g = 0.25, 0.75
    kl, dI, pbar = oracle.indexer_loss(Q, K, idx, sc, scale, g, want_pbar=True)
    tp, I, mask = _torch_teacher_student(Q, K, idx, sc, scale, H)
    np.testing.assert_allclose(_slots_to_dense(pbar, idx, S), tp.numpy(), rtol=1e-12, atol=1e-15)
    I = I.clone().requires_grad_(True)
    logq = torch.log_softmax(I.masked_fill(~mask, float("-inf")), dim=-1)
    # KL(p || q) through torch's kl_div (input log q, target p), zero outside the mask
    terms = torch.nn.functional.kl_div(torch.where(mask, logq, torch.zeros_like(logq)), tp,
                                       reduction="none")
    row_kl = torch.where(mask, terms, torch.zeros_like(terms)).sum(-1)
    np.testing.assert_allclose(kl, row_kl.reshape(-1).detach().numpy(), rtol=1e-11, atol=1e-14)
    (g * row_kl.sum()).backward()
    np.testing.assert_allclose(_slots_to_dense(dI, idx, S), I.grad.numpy(), rtol=1e-10,
                               atol=1e-14)


def test_indexer_loss_two_key_closed_form():
    """One head, two selected keys: Bernoulli KL written with the logistic function."""
    B, S, H, Dqk, k = 1, 6, 1, 8, 2
    Q, K, _, _, _, _, _, _ = _iloss_case(B, S, H, Dqk, seed=42, k=k)
    t, s0, s1 = 5, 1, 4
    idx = np.full((B, S, k), -1, dtype=np.int32)
    idx[0, t] = [s0, s1]
    scores = np.full((B * S, S), np.nan)
    c0, c1 = 0.375, -1.25
    scores[t, s0], scores[t, s1] = c0, c1
    scale, g = 0.5, 2.0
    kl, dI = oracle.indexer_loss(Q, K, idx, scores[t:t + 1], scale, g, rows=np.array([t]))
    qv = bf16_bits_to_f64(Q)[0, t, 0]
    kv = bf16_bits_to_f64(K)[0, :, 0]
    a0, a1 = scale * float(qv @ kv[s0]), scale * float(qv @ kv[s1])
    p = 1.0 / (1.0 + np.exp(a1 - a0))      # teacher weight of s0
    q = 1.0 / (1.0 + np.exp(c1 - c0))      # student weight of s0
    want = p * np.log(p / q) + (1 - p) * np.log((1 - p) / (1 - q))
    assert abs(kl[0] - want) <= 1e-13
    np.testing.assert_allclose(dI[0], [g * (q - p), g * (p - q)], rtol=1e-12, atol=1e-15)


def test_indexer_loss_invariants():
    B, S, H, Dqk, k = 2, 30, 4, 16, 5
    Q, K, _, _, _, _, sc, idx = _iloss_case(B, S, H, Dqk, seed=43, k=k)
    scale = 0.3
    kl, dI, pbar = oracle.indexer_loss(Q, K, idx, sc, scale, 1.0, want_pbar=True)
    assert (kl >= -1e-15).all()
    np.testing.assert_allclose(pbar.sum(axis=1), 1.0, rtol=1e-13)     # every row has key t
    np.testing.assert_allclose(dI.sum(axis=1), 0.0, atol=1e-14)
    # a constant shift of a row's scores changes neither the loss nor its gradient
    kl2, dI2 = oracle.indexer_loss(Q, K, idx, sc + 3.5, scale, 1.0)
    np.testing.assert_allclose(kl2, kl, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(dI2, dI, rtol=1e-10, atol=1e-15)
    # a student equal to the target has zero loss and zero gradient
    st = np.full_like(sc, -np.inf)
    for r in range(B * S):
        for j in range(k):
            s = idx.reshape(-1, k)[r, j]
            if s >= 0 and pbar[r, j] > 0:
                st[r, s] = np.log(pbar[r, j])
    kl3, dI3 = oracle.indexer_loss(Q, K, idx, st, scale, 1.0)
    assert np.max(np.abs(kl3)) < 1e-13 and np.max(np.abs(dI3)) < 1e-15
    # one head: the target is the attention's own softmax weights (exp(l - LSE))
    kl1, dI1, p1 = oracle.indexer_loss(Q[:, :, :1], K, idx, sc, scale, 1.0, want_pbar=True)
    _, lse = oracle.attn_fwd(Q[:, :, :1], K, K[..., :8], idx, scale)
    qv, kv = bf16_bits_to_f64(Q)[:, :, 0], bf16_bits_to_f64(K)[:, :, 0]
    for r in (0, 17, 29, 45):
        b, t = divmod(r, S)
        for j in range(k):
            s = idx[b, t, j]
            if 0 <= s <= t:
                want = np.exp(scale * float(qv[b, t] @ kv[b, s]) - lse[r, 0])
                assert abs(p1[r, j] - want) <= 1e-13


def _torch_indexer_loss(q_idx, k_idx, w, tp, mask, g):
    q = torch.from_numpy(bf16_bits_to_f64(q_idx)).requires_grad_(True)
    kk = torch.from_numpy(bf16_bits_to_f64(k_idx)).requires_grad_(True)
    ww = torch.from_numpy(w.astype(np.float64)).requires_grad_(True)
    z = torch.einsum("bthd,bsd->bths", q, kk)
    I = (ww[..., None] * torch.relu(z)).sum(dim=2)
    logq = torch.log_softmax(I.masked_fill(~mask, float("-inf")), dim=-1)
    safe = torch.where(mask & (tp > 0), tp, torch.ones_like(tp))
    kl = torch.where(mask & (tp > 0), tp * (torch.log(safe) - logq), torch.zeros_like(tp))
    (g * kl.sum()).backward()
    return q.grad.numpy(), kk.grad.numpy(), ww.grad.numpy()


@pytest.mark.parametrize("seg_docs", [0, 2])
def test_indexer_loss_bwd_matches_torch_autograd(seg_docs):
    """Autograd through I = sum_h w relu(q.k) (relu'(0) = 0 in torch too, and the dyadic
    inputs make many z exactly 0) into the KL with a constant target."""
    B, S, H, Dqk, k, Hi, Di = 2, 28, 3, 16, 5, 4, 16
    Q, K, q_idx, k_idx, w, seg, sc, idx = _iloss_case(B, S, H, Dqk, seed=44, k=k, Hi=Hi, Di=Di,
                                                      seg_docs=seg_docs)
    scale, g = 0.4, 1.5
    _, dI = oracle.indexer_loss(Q, K, idx, sc, scale, g)
    dq, dk, dw = oracle.indexer_loss_bwd(q_idx, k_idx, w, idx, dI)
    tp, _, mask = _torch_teacher_student(Q, K, idx, sc, scale, H)
    z = np.einsum("bthd,bsd->bths", bf16_bits_to_f64(q_idx), bf16_bits_to_f64(k_idx))
    assert (z[np.broadcast_to(mask[:, :, None].numpy(), z.shape)] == 0).any()
    gq, gk, gw = _torch_indexer_loss(q_idx, k_idx, w, tp, mask, g)
    np.testing.assert_allclose(dq.reshape(gq.shape), gq, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(dk, gk, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(dw.reshape(gw.shape), gw, rtol=1e-10, atol=1e-13)
    # rows split in two contribute parts of dk that add up
    rows_a, rows_b = np.arange(0, B * S, 2), np.arange(1, B * S, 2)
    _, dka, _ = oracle.indexer_loss_bwd(q_idx, k_idx, w, idx, dI[rows_a], rows=rows_a)
    _, dkb, _ = oracle.indexer_loss_bwd(q_idx, k_idx, w, idx, dI[rows_b], rows=rows_b)
    np.testing.assert_allclose(dka + dkb, dk, rtol=1e-12, atol=1e-14)


def test_indexer_loss_bwd_finite_differences():
    """Central differences of the whole chain q_idx, k_idx, w -> scores -> loss."""
    B, S, H, Dqk, k, Hi, Di = 1, 14, 2, 16, 4, 3, 8
    Q, K, q_idx, k_idx, w, _, sc, idx = _iloss_case(B, S, H, Dqk, seed=45, k=k, Hi=Hi, Di=Di)
    scale, g = 0.5, 1.0
    one = f64_to_bf16_bits(np.array([1.0]))[0]
    arrs = {"q": q_idx.copy(), "k": k_idx.copy(), "w": w.copy()}
    probes = [("q", (0, 11, 1, 2)), ("q", (0, 6, 0, 5)), ("k", (0, 3, 1)), ("k", (0, 9, 6)),
              ("w", (0, 12, 2)), ("w", (0, 8, 0))]
    for name, ix in probes:
        arrs[name][ix] = 1.0 if name == "w" else one
    sc0 = oracle.index_scores(arrs["q"], arrs["k"], arrs["w"], None)
    _, dI = oracle.indexer_loss(Q, K, idx, sc0, scale, g)
    dq, dk, dw = oracle.indexer_loss_bwd(arrs["q"], arrs["k"], arrs["w"], idx, dI)
    grads = {"q": dq.reshape(q_idx.shape), "k": dk, "w": dw.reshape(w.shape)}
    z = np.einsum("bthd,bsd->bths", bf16_bits_to_f64(arrs["q"]), bf16_bits_to_f64(arrs["k"]))
    eps = 2.0 ** -7          # 1 +- 2^-7 are bf16 values; no z of the rows crosses 0 (checked)

    def loss(a):
        s = oracle.index_scores(a["q"], a["k"], a["w"], None)
        kl, _ = oracle.indexer_loss(Q, K, idx, s, scale, g)
        return float(g * kl.sum())

    checked = 0
    for name, ix in probes:
        if name == "q":
            zz = z[0, ix[1], ix[2], : ix[1] + 1]
        elif name == "k":
            zz = z[0, ix[1]:, :, ix[1]]
        else:
            zz = np.ones(1)
        if (zz == 0).any():
            continue
        vals = []
        for sgn in (+1, -1):
            a = {n: x.copy() for n, x in arrs.items()}
            a[name][ix] = (1.0 + sgn * eps) if name == "w" else \
                f64_to_bf16_bits(np.array([1.0 + sgn * eps]))[0]
            vals.append(loss(a))
        fd = (vals[0] - vals[1]) / (2 * eps)
        an = grads[name][ix]
        assert abs(fd - an) <= 2e-3 * max(1e-2, abs(an)), (name, ix, fd, an)
        checked += 1
    assert checked >= 4
