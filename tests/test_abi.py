"""The C ABI loads without a GPU, exports every declared symbol, and rejects bad
arguments on the host before anything is launched (no device is touched)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dsa():
    import __graft_entry__
    __graft_entry__.build()
    import sparse_attention_index_gb300 as m
    return m


def _declared():
    text = open(os.path.join(ROOT, "include", "dsa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"\b(dsa_[a-z0-9_]+)\s*\(", text))


def test_every_declared_symbol_is_exported(dsa):
    declared = _declared()
    assert declared == set(dsa.EXPORTS)
    for name in declared:
        assert hasattr(dsa.lib, name), name


def test_status_strings_and_version(dsa):
    assert dsa.lib.dsa_status_string(0) == b"DSA_OK"
    assert dsa.lib.dsa_status_string(2) == b"DSA_ERR_UNSUPPORTED"
    assert dsa.lib.dsa_status_string(99) == b"DSA_ERR_UNKNOWN"
    assert dsa.lib.dsa_version() == 100


def _r256(n):
    return (n + 255) // 256 * 256


def test_workspace_sizes(dsa):
    """The attention workspaces hold the fp32 dK / dV accumulators and, wherever the
    dense-tile kernels can take the shape, their bitmap [B*S, 4*QT] uint32, tile flags
    [B, QT, QT] bytes and (backward) Delta [B*S, H] fp32, each on a 256-byte boundary."""
    B, S, H = 1, 16384, 128
    QT = S // 128
    bits, flags, delta = B * S * QT * 16, B * QT * QT, B * S * H * 4
    dense_fwd = _r256(bits) + _r256(flags)
    dense_bwd = dense_fwd + _r256(delta)
    acc = B * S * 320 * 4
    assert dsa.lib.dsa_sparse_attn_fwd_workspace_size(B, S, H, 1, 192, 128) == dense_fwd
    assert dsa.lib.dsa_sparse_attn_bwd_workspace_size(B, S, H, 1, 192, 128) == acc + dense_bwd
    # per-head K / V: accumulators per K / V head
    assert dsa.lib.dsa_sparse_attn_bwd_workspace_size(1, 4096, 128, 128, 192, 128) == \
        4096 * 128 * 320 * 4 + _r256(4096 * 32 * 16) + _r256(32 * 32) + _r256(4096 * 128 * 4)
    # no dense-tile kernel for these shapes: nothing reserved for it
    assert dsa.lib.dsa_sparse_attn_fwd_workspace_size(1, 131072, 128, 1, 192, 128) == 0
    assert dsa.lib.dsa_sparse_attn_fwd_workspace_size(1, 128, 2, 1, 32, 32) == 0
    assert dsa.lib.dsa_sparse_attn_bwd_workspace_size(1, 128, 2, 1, 32, 32) == _r256(128 * 64 * 4)
    assert dsa.lib.dsa_sparse_attn_bwd_workspace_size(0, 1, 1, 1, 1, 1) == 0
    assert dsa.lib.dsa_topk_workspace_size(1, 16384, 2048) == 0


# Fake (never dereferenced) 16-byte-aligned addresses: every call below fails
# validation on the host and returns before any CUDA call.
P = ctypes.c_void_p(1 << 20)
MIS = ctypes.c_void_p((1 << 20) + 4)


def test_index_scores_validation(dsa):
    f = dsa.lib.dsa_index_scores
    assert f(None, P, P, 1, None, 1, 128, 64, 128, P, 128, None) == 1        # null q_idx
    assert f(P, P, P, 1, None, 1, 128, 64, 128, P, 100, None) == 1           # ld < S
    assert f(P, P, P, 1, None, 1, 128, 64, 128, P, 130, None) == 1           # ld % 4
    assert f(P, P, P, 7, None, 1, 128, 64, 128, P, 128, None) == 1           # bad w dtype
    assert f(MIS, P, P, 1, None, 1, 128, 64, 128, P, 128, None) == 1         # misaligned
    assert f(P, P, P, 1, None, 0, 128, 64, 128, P, 128, None) == 1           # B = 0
    assert f(P, P, P, 1, None, 1, 128, 48, 128, P, 128, None) == 2           # Hi not 2^n
    assert f(P, P, P, 1, None, 1, 128, 64, 96, P, 128, None) == 2            # Di unsupported
    assert f(P, P, P, 1, None, 1, 128, 256, 128, P, 128, None) == 2          # Hi > 128


def test_topk_validation(dsa):
    f = dsa.lib.dsa_topk
    # scores, ld, seg, B, S, k, idx, count, vals, ws, ws_bytes, stream
    assert f(None, 128, None, 1, 128, 4, P, None, None, None, 0, None) == 1
    assert f(P, 127, None, 1, 128, 4, P, None, None, None, 0, None) == 1
    assert f(P, 128, None, 1, 128, 0, P, None, None, None, 0, None) == 1
    assert f(P, 128, MIS, 1, 128, 4, P, None, None, None, 0, None) == 1
    assert f(P, 128, None, 1, 128, 4, P, None, MIS, None, 0, None) == 1        # vals misaligned


def test_attention_validation(dsa):
    fwd = dsa.lib.dsa_sparse_attn_fwd
    fneed = dsa.lib.dsa_sparse_attn_fwd_workspace_size(1, 64, 16, 1, 192, 128)
    assert fneed > 0
    W = (P, fneed)
    # B, S, H, Hkv, Dqk, Dv, k
    assert fwd(P, P, P, P, 1, 64, 16, 1, 192, 128, 8, 0.1, None, P, *W, None) == 1   # null O
    assert fwd(P, P, P, P, 1, 64, 16, 3, 192, 128, 8, 0.1, P, P, *W, None) == 1      # H % Hkv
    # per-head K / V runs on the dense-tile kernels only, which take (192, 128) / (128, 128)
    assert fwd(P, P, P, P, 1, 64, 16, 16, 64, 64, 8, 0.1, P, P, *W, None) == 2       # Hkv = H, 64
    assert fwd(P, P, P, P, 1, 70000, 16, 16, 192, 128, 8, 0.1, P, P, *W, None) == 2  # Hkv = H, S
    assert fwd(P, P, P, P, 1, 64, 256, 1, 192, 128, 8, 0.1, P, P, *W, None) == 2     # H > 128
    assert fwd(P, P, P, P, 1, 64, 16, 1, 96, 128, 8, 0.1, P, P, *W, None) == 2       # dims
    assert fwd(P, P, P, P, 1, 64, 16, 1, 100, 128, 8, 0.1, P, P, *W, None) == 1      # Dqk % 16
    # the dense-tile kernel's bitmap is the caller's: refused without it, whichever kernel
    assert fwd(P, P, P, P, 1, 64, 16, 1, 192, 128, 8, 0.1, P, P, None, fneed, None) == 3
    assert fwd(P, P, P, P, 1, 64, 16, 1, 192, 128, 8, 0.1, P, P, P, fneed - 1, None) == 3
    assert fwd(P, P, P, P, 1, 64, 16, 1, 192, 128, 8, 0.1, P, P, MIS, fneed, None) == 3
    assert dsa.lib.dsa_sparse_attn_fwd_dense(P, P, P, P, 1, 64, 16, 4, 192, 128, 8, 0.1, P, P,
                                             None, 0, None) == 3
    bwd = dsa.lib.dsa_sparse_attn_bwd
    need = dsa.lib.dsa_sparse_attn_bwd_workspace_size(1, 64, 16, 1, 192, 128)
    assert need == _r256(64 * 320 * 4) + fneed + _r256(64 * 16 * 4)
    args = [P] * 7 + [1, 64, 16, 1, 192, 128, 8, 0.1] + [P, P, P]
    assert bwd(*args, None, need, None) == 3                                      # no ws
    assert bwd(*args, P, need - 4, None) == 3                                     # small ws
    assert bwd(*args, MIS, need, None) == 3                                       # misaligned
    assert bwd(*([P] * 6 + [None] + args[7:]), P, need, None) == 1                # null dO
    assert dsa.lib.dsa_sparse_attn_bwd_dense(*args, P, need - 256, None) == 3
    # the no-allocation backward: the same argument checks, then its own limits
    na = dsa.lib.dsa_sparse_attn_bwd_noalloc
    assert na(*([P] * 6 + [None] + args[7:]), None) == 1                          # null dO
    assert na(*([P] * 7 + [1, 64, 16, 1, 100, 128, 8, 0.1] + [P, P, P]), None) == 1  # Dqk % 16
    assert na(*([P] * 7 + [1, 64, 256, 1, 192, 128, 8, 0.1] + [P, P, P]), None) == 2  # H > 128
    assert na(*([P] * 7 + [1, 64, 16, 16, 192, 128, 8, 0.1] + [P, P, P]), None) == 2  # Hkv > 1
    assert na(*([P] * 7 + [1, 40000, 16, 1, 192, 128, 8, 0.1] + [P, P, P]), None) == 3  # limit


def test_index_topk_validation(dsa):
    """The fused indexer + top-k: its workspace is one block of query rows, and bad
    arguments are refused before anything is launched."""
    assert dsa.lib.dsa_index_topk_workspace_size(1, 131072, 2048) == 2048 * 131072 * 4
    assert dsa.lib.dsa_index_topk_workspace_size(2, 489, 2048) == 2 * 489 * 492 * 4   # S < block
    assert dsa.lib.dsa_index_topk_workspace_size(0, 128, 256) == 0
    f = dsa.lib.dsa_index_topk
    need = dsa.lib.dsa_index_topk_workspace_size(1, 1024, 256)
    # q_idx, k_idx, w, w_dtype, seg, B, S, Hi, Di, k, block_rows, idx, count, vals, ws,
    # ws_bytes, stream
    A = (1, None, 1, 1024, 64, 128, 8, 256, P, P)
    assert f(None, P, P, *A, None, P, need, None) == 1                                # null q_idx
    assert f(P, P, P, 1, None, 1, 1024, 64, 128, 8, 100, P, P, None, P, need, None) == 1  # block
    assert f(P, P, P, 1, None, 1, 1024, 64, 128, 0, 256, P, P, None, P, need, None) == 1  # k = 0
    assert f(P, P, P, 1, None, 1, 1024, 48, 128, 8, 256, P, P, None, P, need, None) == 2  # Hi
    assert f(P, P, P, *A, MIS, P, need, None) == 1                                    # vals
    assert f(P, P, P, *A, None, P, need - 16, None) == 3                              # small ws
    assert f(P, P, P, *A, None, None, need, None) == 3                                # no ws


def test_index_topk_fp8_validation(dsa):
    """The e4m3 form of the fused indexer + top-k refuses the same bad arguments, plus a
    misaligned key scale and an index head dim that is not a multiple of 16."""
    f = dsa.lib.dsa_index_topk_fp8
    need = dsa.lib.dsa_index_topk_workspace_size(1, 1024, 256)
    # q_idx, k_idx, k_scale, w, w_dtype, seg, B, S, Hi, Di, k, block_rows, idx, count, vals,
    # ws, ws_bytes, stream
    assert f(None, P, None, P, 1, None, 1, 1024, 64, 128, 8, 256, P, P, None, P, need, None) == 1
    odd = ctypes.c_void_p((1 << 20) + 4)   # k_scale not on a 16-byte boundary
    assert f(P, P, odd, P, 1, None, 1, 1024, 64, 128, 8, 256, P, P, None, P, need, None) == 1
    assert f(P, P, None, P, 1, None, 1, 1024, 64, 40, 8, 256, P, P, None, P, need, None) == 1
    assert f(P, P, None, P, 1, None, 1, 1024, 64, 128, 8, 100, P, P, None, P, need, None) == 1
    assert f(P, P, None, P, 1, None, 1, 1024, 48, 128, 8, 256, P, P, None, P, need, None) == 2
    assert f(P, P, None, P, 1, None, 1, 1024, 64, 128, 8, 256, P, P, None, P, need - 16,
             None) == 3


def test_index_topk_stream_validation(dsa):
    """The streaming form refuses bad arguments before any launch: its selected scores
    (vals) are staged by slot, so they need k <= 2048."""
    f = dsa.lib.dsa_index_topk_stream
    need = dsa.lib.dsa_index_topk_stream_workspace_size(1, 8192, 1024)
    assert need > 0
    # q_idx, k_idx, w, w_dtype, seg, B, S, Hi, Di, k, block_rows, idx, count, vals, ws,
    # ws_bytes, stream
    assert f(P, P, P, 1, None, 1, 8192, 64, 128, 4096, 1024, P, P, P, P, need, None) == 2
    assert f(P, P, P, 1, None, 1, 8192, 64, 128, 2048, 1024, P, P, MIS, P, need, None) == 1
    assert f(P, P, P, 1, None, 1, 200000, 64, 128, 2048, 1024, P, P, None, P, need, None) == 2
    assert f(P, P, P, 1, None, 1, 8192, 64, 128, 2048, 1024, P, P, P, P, need - 16, None) == 3
    assert dsa.lib.dsa_index_topk_stream_fp8(P, P, None, P, 1, None, 1, 8192, 64, 128, 4096,
                                             1024, P, P, P, P, need, None) == 2


def test_indexer_loss_validation(dsa):
    """The loss reads the scores by key (ld_scores >= S) or the top-k's selected scores by
    slot (ld_scores = 0); other strides are refused before any launch."""
    f = dsa.lib.dsa_indexer_loss
    # Q, K, idx, lse, scores, ld, B, S, H, Hkv, Dqk, k, scale, grad_scale, kl, dI, stream
    assert f(P, P, P, P, P, -4, 1, 128, 16, 1, 128, 8, 0.1, 1.0, P, P, None) == 1
    assert f(P, P, P, P, P, 64, 1, 128, 16, 1, 128, 8, 0.1, 1.0, P, P, None) == 1
    assert f(P, P, P, P, None, 0, 1, 128, 16, 1, 128, 8, 0.1, 1.0, P, P, None) == 1
