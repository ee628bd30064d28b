"""fp64 CPU oracle for the DSA layer hot path (test infrastructure).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the library's product
path never does. It shares no code with the CUDA sources. The arithmetic lives
in ``dsa_oracle.c`` (plain C, fp64, POSIX threads over query rows); this module
compiles it with gcc and marshals numpy arrays.

Functions and the passages they follow (details in ``dsa_oracle.c``):

* ``index_scores`` - indexer score, "DeepSeek3.2: Onboard sparse attention"
  (Background: per-head qk product) and "Implement QK attention head chunking
  for CSA" (Description: per-head products reduced over heads), causal and
  document mask from "Support Ring Attention with DeepSeek DSA Sparse Indexer"
  (Forward Flow step 3).
* ``index_scores_fp8`` / ``e4m3_decode`` - the indexer score from OCP FP8 E4M3
  inputs with a per-key scale of k ("DeepSeek3.2: Onboard sparse attention",
  What this PR does item 4: the original indexer is an fp8 kernel).
* ``topk`` - per-query top-k index selection, ties to the lower index
  ("DeepSeek3.2: Onboard sparse attention", Background).
* ``attn_fwd`` / ``attn_bwd`` - masked softmax attention over the selected
  keys and its gradients ("Support Ring Attention with DeepSeek DSA Sparse
  Indexer", Forward Flow step 5, Backward Flow step 6).
* ``indexer_loss`` / ``indexer_loss_bwd`` - the indexer's auxiliary loss: a
  head-summed fp32 softmax target of the attention scores over the valid
  tokens, held constant ("Implement QK attention head chunking for CSA", the
  indexer-loss teacher), added to the objective so that its gradient trains
  the indexer ("Support Ring Attention with DeepSeek DSA Sparse Indexer", Loss
  Harvesting & Objective Injection); KL form and normalisation as read in
  ``dsa_oracle.c``.

Pins (tests/test_oracle_pins.py): exact rational arithmetic, brute-force
sorting, dense masked attention through torch in fp64, autograd and finite
differences, and invariants. No function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``liboracle.so`` (gcc -O2, strict IEEE fp64)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                    "-ffp-contract=off", "-o", tmp, _SRC, "-lm", "-lpthread"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, ci, i64, cd = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_index_scores.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, vp, i64, vp, ci]
            lib.oracle_index_scores.restype = None
            lib.oracle_index_scores_fp8.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, vp, i64,
                                                    vp, ci]
            lib.oracle_index_scores_fp8.restype = None
            lib.oracle_e4m3_decode.argtypes = [vp, i64, vp]
            lib.oracle_e4m3_decode.restype = None
            lib.oracle_topk.argtypes = [vp, vp, ci, ci, vp, i64, vp, vp, ci]
            lib.oracle_topk.restype = None
            lib.oracle_attn_fwd.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, cd, vp,
                                            i64, vp, vp, ci]
            lib.oracle_attn_fwd.restype = ci
            lib.oracle_attn_bwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, cd,
                                            vp, i64, vp, vp, vp, ci]
            lib.oracle_attn_bwd.restype = ci
            lib.oracle_indexer_loss.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cd, cd,
                                                vp, i64, vp, vp, vp, ci]
            lib.oracle_indexer_loss.restype = ci
            lib.oracle_indexer_loss_bwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, vp,
                                                    i64, vp, vp, vp, ci]
            lib.oracle_indexer_loss_bwd.restype = ci
            _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


def _rows(rows, B, S):
    if rows is None:
        rows = np.arange(B * S, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    if rows.size and (rows.min() < 0 or rows.max() >= B * S):
        raise ValueError("row out of range")
    return rows


def index_scores(q_idx, k_idx, w, seg, rows=None, threads=None) -> np.ndarray:
    """q_idx [B,S,Hi,Di] (uint16 bf16 bits), k_idx [B,S,Di], w [B,S,Hi] f32, seg [B,S] or None.

    Returns fp64 [len(rows), S]: s <= t -> score or -inf (other document), s > t -> NaN.
    """
    B, S, Hi, Di = q_idx.shape
    assert k_idx.shape == (B, S, Di) and w.shape == (B, S, Hi)
    q, qp = _c(q_idx, np.uint16)
    k, kp = _c(k_idx, np.uint16)
    ww, wp = _c(w, np.float32)
    sp = None
    if seg is not None:
        sg, sp = _c(seg, np.int32)
    rows = _rows(rows, B, S)
    out = np.empty((rows.size, S), dtype=np.float64)
    _load().oracle_index_scores(qp, kp, wp, sp, B, S, Hi, Di, rows.ctypes.data, rows.size,
                                out.ctypes.data, threads or default_threads())
    return out


def e4m3_decode(b) -> np.ndarray:
    """OCP FP8 E4M3 bytes (uint8, any shape) -> their exact fp64 values (NaN for S.1111.111)."""
    a, ap = _c(b, np.uint8)
    out = np.empty(a.shape, dtype=np.float64)
    _load().oracle_e4m3_decode(ap, a.size, out.ctypes.data)
    return out


def index_scores_fp8(q8, k8, w, seg, k_scale=None, rows=None, threads=None) -> np.ndarray:
    """q8 [B,S,Hi,Di], k8 [B,S,Di] e4m3 bytes, w [B,S,Hi] f32, seg [B,S] or None, k_scale [B,S].

    Same output convention as ``index_scores``.
    """
    B, S, Hi, Di = q8.shape
    assert k8.shape == (B, S, Di) and w.shape == (B, S, Hi)
    q, qp = _c(q8, np.uint8)
    k, kp = _c(k8, np.uint8)
    ww, wp = _c(w, np.float32)
    sp = cp = None
    if seg is not None:
        sg, sp = _c(seg, np.int32)
    if k_scale is not None:
        ks, cp = _c(k_scale, np.float32)
    rows = _rows(rows, B, S)
    out = np.empty((rows.size, S), dtype=np.float64)
    _load().oracle_index_scores_fp8(qp, kp, cp, wp, sp, B, S, Hi, Di, rows.ctypes.data, rows.size,
                                    out.ctypes.data, threads or default_threads())
    return out


def topk(scores, seg, S: int, k: int, rows=None, B: int = 1, threads=None):
    """scores [len(rows), S] (any float; only s <= t read). Returns (idx [n,k] int32, count [n])."""
    rows = _rows(rows, B, S)
    sc, scp = _c(scores, np.float64)
    assert sc.shape == (rows.size, S)
    sp = None
    if seg is not None:
        sg, sp = _c(seg, np.int32)
    idx = np.empty((rows.size, k), dtype=np.int32)
    cnt = np.empty((rows.size,), dtype=np.int32)
    _load().oracle_topk(scp, sp, S, k, rows.ctypes.data, rows.size, idx.ctypes.data,
                        cnt.ctypes.data, threads or default_threads())
    return idx, cnt


def attn_fwd(Q, K, V, idx, scale: float, rows=None, threads=None):
    """Q [B,S,H,Dqk], K [B,S,Hkv,Dqk], V [B,S,Hkv,Dv] (bf16 bits), idx [B,S,k].

    Returns (O [n,H,Dv] fp64, lse [n,H] fp64) for the listed rows.
    """
    B, S, H, Dqk = Q.shape
    Hkv, Dv = V.shape[2], V.shape[3]
    k = idx.shape[2]
    q, qp = _c(Q, np.uint16)
    kk, kp = _c(K, np.uint16)
    v, vp = _c(V, np.uint16)
    ix, ip = _c(idx, np.int32)
    rows = _rows(rows, B, S)
    O = np.empty((rows.size, H, Dv), dtype=np.float64)
    lse = np.empty((rows.size, H), dtype=np.float64)
    rc = _load().oracle_attn_fwd(qp, kp, vp, ip, B, S, H, Hkv, Dqk, Dv, k, float(scale),
                                 rows.ctypes.data, rows.size, O.ctypes.data, lse.ctypes.data,
                                 threads or default_threads())
    if rc:
        raise ValueError(f"oracle_attn_fwd: bad input (code {rc})")
    return O, lse


def attn_bwd(Q, K, V, idx, dO, scale: float, rows=None, threads=None):
    """Returns (dQ [n,H,Dqk], dK [B,S,Hkv,Dqk], dV [B,S,Hkv,Dv]) in fp64.

    dK / dV hold the contributions of the listed rows (all rows: full gradient).
    """
    B, S, H, Dqk = Q.shape
    Hkv, Dv = V.shape[2], V.shape[3]
    k = idx.shape[2]
    q, qp = _c(Q, np.uint16)
    kk, kp = _c(K, np.uint16)
    v, vp = _c(V, np.uint16)
    d, dp = _c(dO, np.uint16)
    ix, ip = _c(idx, np.int32)
    rows = _rows(rows, B, S)
    dQ = np.empty((rows.size, H, Dqk), dtype=np.float64)
    dK = np.empty((B, S, Hkv, Dqk), dtype=np.float64)
    dV = np.empty((B, S, Hkv, Dv), dtype=np.float64)
    rc = _load().oracle_attn_bwd(qp, kp, vp, ip, dp, B, S, H, Hkv, Dqk, Dv, k, float(scale),
                                 rows.ctypes.data, rows.size, dQ.ctypes.data, dK.ctypes.data,
                                 dV.ctypes.data, threads or default_threads())
    if rc:
        raise ValueError(f"oracle_attn_bwd: bad input (code {rc})")
    return dQ, dK, dV


def indexer_loss(Q, K, idx, scores, scale: float, grad_scale: float = 1.0, rows=None,
                 threads=None, want_pbar: bool = False):
    """Q [B,S,H,Dqk], K [B,S,Hkv,Dqk] (bf16 bits), idx [B,S,k], scores [n,S] (any float).

    Returns (kl [n], dI [n,k]) in fp64, plus pbar [n,k] (the target) if asked.
    """
    B, S, H, Dqk = Q.shape
    Hkv = K.shape[2]
    k = idx.shape[2]
    q, qp = _c(Q, np.uint16)
    kk, kp = _c(K, np.uint16)
    ix, ip = _c(idx, np.int32)
    rows = _rows(rows, B, S)
    sc, sp = _c(scores, np.float64)
    if sc.shape != (rows.size, S):
        raise ValueError("scores must be [len(rows), S]")
    kl = np.empty((rows.size,), dtype=np.float64)
    dI = np.empty((rows.size, k), dtype=np.float64)
    pbar = np.empty((rows.size, k), dtype=np.float64) if want_pbar else None
    rc = _load().oracle_indexer_loss(qp, kp, ip, sp, B, S, H, Hkv, Dqk, k, float(scale),
                                     float(grad_scale), rows.ctypes.data, rows.size,
                                     kl.ctypes.data, dI.ctypes.data,
                                     pbar.ctypes.data if want_pbar else None,
                                     threads or default_threads())
    if rc:
        raise ValueError(f"oracle_indexer_loss: bad input (code {rc})")
    return (kl, dI, pbar) if want_pbar else (kl, dI)


def indexer_loss_bwd(q_idx, k_idx, w, idx, dI, rows=None, threads=None):
    """q_idx [B,S,Hi,Di], k_idx [B,S,Di] (bf16 bits), w [B,S,Hi] f32, idx [B,S,k], dI [n,k].

    Returns (dq [n,Hi,Di], dk [B,S,Di], dw [n,Hi]) in fp64; dk holds the listed rows'
    contributions (all rows: the full gradient).
    """
    B, S, Hi, Di = q_idx.shape
    k = idx.shape[2]
    q, qp = _c(q_idx, np.uint16)
    kk, kp = _c(k_idx, np.uint16)
    ww, wp = _c(w, np.float32)
    ix, ip = _c(idx, np.int32)
    rows = _rows(rows, B, S)
    g, gp = _c(dI, np.float64)
    if g.shape != (rows.size, k):
        raise ValueError("dI must be [len(rows), k]")
    dq = np.empty((rows.size, Hi, Di), dtype=np.float64)
    dk = np.empty((B, S, Di), dtype=np.float64)
    dw = np.empty((rows.size, Hi), dtype=np.float64)
    rc = _load().oracle_indexer_loss_bwd(qp, kp, wp, ip, gp, B, S, Hi, Di, k, rows.ctypes.data,
                                         rows.size, dq.ctypes.data, dk.ctypes.data,
                                         dw.ctypes.data, threads or default_threads())
    if rc:
        raise ValueError(f"oracle_indexer_loss_bwd: bad input (code {rc})")
    return dq, dk, dw
