"""dsa_sparse_attn_bwd_noalloc, the backward for callers that cannot allocate.

Such callers (a plugin whose host runtime owns every device allocation, or code
that must not call cudaMalloc while it runs) cannot pass the fp32 workspace of
dsa_sparse_attn_bwd. The variant keeps that accumulator in a fixed array inside
the library. These tests call it through the C ABI and compare it with the
workspace entry point and with the fp64 oracle, twice in a row, since every
call reuses the same array.
This file is collected last so that a failure here stops a -x run only after
every other test has run; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TOL, bf16_dev, dev, host_f64, rel_err

pytestmark = pytest.mark.gpu


def _host_inputs(B, S, H, Dqk, Dv, k, seed):
    Q = synth.normal_bf16((B, S, H, Dqk), seed, synth.STREAM_Q)
    K = synth.normal_bf16((B, S, 1, Dqk), seed, synth.STREAM_K)
    V = synth.normal_bf16((B, S, 1, Dv), seed, synth.STREAM_V)
    dO = synth.normal_bf16((B, S, H, Dv), seed, synth.STREAM_DO)
    q_idx = synth.dyadic_bf16((B, S, 4, 32), seed, synth.STREAM_Q_IDX, -8, 8, 3)
    k_idx = synth.dyadic_bf16((B, S, 32), seed, synth.STREAM_K_IDX, -8, 8, 3)
    w = synth.dyadic_f32((B, S, 4), seed, synth.STREAM_W, -1, 1, 4)
    sc = oracle.index_scores(q_idx, k_idx, w, None)
    idx, _ = oracle.topk(sc, None, S, k, B=B)
    return Q, K, V, dO, idx.reshape(B, S, k)


@pytest.mark.parametrize("shape", [(1, 300, 128, 192, 128, 64), (2, 200, 16, 192, 128, 100),
                                   (1, 130, 32, 64, 64, 33)])
def test_noalloc_matches_workspace_entry_point(shape):
    import sparse_attention_index_gb300 as dsa
    B, S, H, Dqk, Dv, k = shape
    hQ, hK, hV, hdO, hidx = _host_inputs(*shape, seed=900 + S)
    Q, K, V, dO, idx = bf16_dev(hQ), bf16_dev(hK), bf16_dev(hV), bf16_dev(hdO), dev(hidx)
    scale = 1.0 / np.sqrt(Dqk)
    O, lse = dsa.dsa_sparse_attn_fwd(Q, K, V, idx, scale)
    ref = dsa.dsa_sparse_attn_bwd(Q, K, V, idx, O, lse, dO, scale)
    # and the fp64 oracle's gradients of the same selection
    dQ_o, dK_o, dV_o = oracle.attn_bwd(hQ, hK, hV, hidx, hdO, scale)
    oracle_ref = (dQ_o.reshape(B, S, H, Dqk), dK_o, dV_o)
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):   # the second call must not see what the first left in the array
        dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
        rc = dsa.lib.dsa_sparse_attn_bwd_noalloc(
            Q.data_ptr(), K.data_ptr(), V.data_ptr(), idx.data_ptr(), O.data_ptr(),
            lse.data_ptr(), dO.data_ptr(), B, S, H, 1, Dqk, Dv, k, ctypes.c_float(scale),
            dQ.data_ptr(), dK.data_ptr(), dV.data_ptr(), stream)
        assert rc == 0, dsa.lib.dsa_status_string(rc)
        torch.cuda.synchronize()
        assert dsa.dsa_get_last_device_error() == 0
        for got, want, want_o in zip((dQ, dK, dV), ref, oracle_ref):
            assert rel_err(host_f64(got), host_f64(want)) <= TOL
            assert rel_err(host_f64(got), want_o) <= TOL


def test_noalloc_rejects_sizes_beyond_its_array():
    import sparse_attention_index_gb300 as dsa
    # B*S*(Dqk+Dv) = 1 * 40000 * 320 > 8388608 floats: refused before any launch
    t = torch.zeros(16, dtype=torch.uint8, device="cuda")
    p = t.data_ptr()
    rc = dsa.lib.dsa_sparse_attn_bwd_noalloc(p, p, p, p, p, p, p, 1, 40000, 16, 1, 192, 128, 64,
                                             ctypes.c_float(0.1), p, p, p,
                                             torch.cuda.current_stream().cuda_stream)
    assert rc == 3   # DSA_ERR_WORKSPACE
