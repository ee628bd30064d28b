"""DeepSeek Sparse Attention (DSA) layer hot path for one GB300 (sm_103a).

A thin ctypes binding over ``libdsa.so`` (the C ABI in ``include/dsa.h``).
Every function here only checks tensors and marshals pointers; all the work
runs in the library's CUDA kernels. PyTorch provides device memory and
streams. If the library has not been built the import fails: there is no
fallback path.

Entry points (same names as the C ABI):

* ``dsa_index_scores`` - lightning-indexer scores I[b,t,s] (causal / document mask)
* ``dsa_index_scores_fp8`` - the same from e4m3 q_idx / k_idx, optional per-key scale
* ``dsa_topk``         - per-query top-k key indices, ascending, -1 padded
* ``dsa_sparse_attn_fwd`` - attention over the selected keys -> (O, lse)
* ``dsa_sparse_attn_fwd_dense`` - the same from the dense-tile kernel only
* ``dsa_sparse_attn_bwd`` - its gradients -> (dQ, dK, dV)
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdsa.so")

DSA_BF16, DSA_F32 = 0, 1
# device error codes (dsa_get_last_device_error): kind | stage
DSA_DEVERR_TIMEOUT, DSA_DEVERR_BAD_INDEX, DSA_DEVERR_MISALIGNED = 0x01, 0x02, 0x03
DSA_STAGE_INDEXER, DSA_STAGE_TOPK, DSA_STAGE_FWD, DSA_STAGE_BWD = 0x100, 0x200, 0x300, 0x400
DSA_STAGE_LOSS, DSA_STAGE_LOSS_BWD = 0x500, 0x600
DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED = 0, 1, 2
STATUS = {0: "DSA_OK", 1: "DSA_ERR_INVALID_ARG", 2: "DSA_ERR_UNSUPPORTED", 3: "DSA_ERR_WORKSPACE",
          4: "DSA_ERR_CUDA", 5: "DSA_ERR_TIMEOUT", 6: "DSA_ERR_DEVICE"}

# every symbol include/dsa.h declares
EXPORTS = ("dsa_status_string", "dsa_version", "dsa_get_last_device_error", "dsa_index_scores",
           "dsa_index_scores_fp8",
           "dsa_topk_workspace_size", "dsa_topk", "dsa_sparse_attn_fwd_workspace_size",
           "dsa_sparse_attn_fwd", "dsa_sparse_attn_fwd_dense",
           "dsa_sparse_attn_fwd_kernel", "dsa_sparse_attn_bwd_dense", "dsa_sparse_attn_bwd_kernel",
           "dsa_sparse_attn_bwd_workspace_size", "dsa_sparse_attn_bwd",
           "dsa_sparse_attn_bwd_noalloc", "dsa_indexer_loss", "dsa_indexer_loss_bwd",
           "dsa_index_topk_workspace_size", "dsa_index_topk", "dsa_index_topk_fp8",
           "dsa_index_topk_stream_workspace_size", "dsa_index_topk_stream",
           "dsa_index_topk_stream_fp8")


class DsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS.get(status, status)}")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, ci, i64, sz, cf = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                           ctypes.c_float)
    lib.dsa_status_string.argtypes = [ci]
    lib.dsa_status_string.restype = ctypes.c_char_p
    lib.dsa_version.restype = ci
    lib.dsa_get_last_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
    lib.dsa_index_scores.argtypes = [vp, vp, vp, ci, vp, ci, ci, ci, ci, vp, i64, vp]
    lib.dsa_index_scores_fp8.argtypes = [vp, vp, vp, vp, ci, vp, ci, ci, ci, ci, vp, i64, vp]
    lib.dsa_topk_workspace_size.argtypes = [ci, ci, ci]
    lib.dsa_topk_workspace_size.restype = sz
    lib.dsa_topk.argtypes = [vp, i64, vp, ci, ci, ci, vp, vp, vp, vp, sz, vp]
    lib.dsa_sparse_attn_fwd_workspace_size.argtypes = [ci, ci, ci, ci, ci, ci]
    lib.dsa_sparse_attn_fwd_workspace_size.restype = sz
    lib.dsa_sparse_attn_fwd.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, cf, vp, vp, vp,
                                        sz, vp]
    lib.dsa_sparse_attn_fwd_dense.argtypes = lib.dsa_sparse_attn_fwd.argtypes
    lib.dsa_sparse_attn_fwd_kernel.argtypes = [ci, ci, ci, ci, ci, ci, ci, cf]
    lib.dsa_sparse_attn_fwd_kernel.restype = ci
    lib.dsa_sparse_attn_bwd_kernel.argtypes = [ci, ci, ci, ci, ci, ci, ci, cf]
    lib.dsa_sparse_attn_bwd_kernel.restype = ci
    lib.dsa_sparse_attn_bwd_workspace_size.argtypes = [ci, ci, ci, ci, ci, ci]
    lib.dsa_sparse_attn_bwd_workspace_size.restype = sz
    lib.dsa_sparse_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, cf,
                                        vp, vp, vp, vp, sz, vp]
    lib.dsa_sparse_attn_bwd_dense.argtypes = lib.dsa_sparse_attn_bwd.argtypes
    lib.dsa_sparse_attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci,
                                                ci, ci, cf, vp, vp, vp, vp]
    lib.dsa_indexer_loss.argtypes = [vp, vp, vp, vp, vp, i64, ci, ci, ci, ci, ci, ci, cf, cf, vp,
                                     vp, vp]
    lib.dsa_indexer_loss_bwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, vp, vp, vp, vp]
    lib.dsa_index_topk_workspace_size.argtypes = [ci, ci, ci]
    lib.dsa_index_topk_workspace_size.restype = sz
    lib.dsa_index_topk.argtypes = [vp, vp, vp, ci, vp, ci, ci, ci, ci, ci, ci, vp, vp, vp, vp, sz,
                                   vp]
    lib.dsa_index_topk_fp8.argtypes = [vp, vp, vp, vp, ci, vp, ci, ci, ci, ci, ci, ci, vp, vp, vp,
                                       vp, sz, vp]
    lib.dsa_index_topk_stream_workspace_size.argtypes = [ci, ci, ci]
    lib.dsa_index_topk_stream_workspace_size.restype = sz
    lib.dsa_index_topk_stream.argtypes = lib.dsa_index_topk.argtypes
    lib.dsa_index_topk_stream_fp8.argtypes = lib.dsa_index_topk_fp8.argtypes
    for name in ("dsa_get_last_device_error", "dsa_index_scores", "dsa_index_scores_fp8", "dsa_topk",
                 "dsa_indexer_loss", "dsa_indexer_loss_bwd", "dsa_index_topk",
                 "dsa_index_topk_fp8", "dsa_index_topk_stream", "dsa_index_topk_stream_fp8",
                 "dsa_sparse_attn_fwd", "dsa_sparse_attn_fwd_dense", "dsa_sparse_attn_bwd",
                 "dsa_sparse_attn_bwd_dense", "dsa_sparse_attn_bwd_noalloc"):
        getattr(lib, name).restype = ci
    return lib


lib = _load()


def _check(rc: int, where: str):
    if rc != 0:
        raise DsaError(rc, where)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def dsa_get_last_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error word."""
    code = ctypes.c_int32(0)
    _check(lib.dsa_get_last_device_error(_stream(stream), ctypes.byref(code)),
           "dsa_get_last_device_error")
    return int(code.value)


def dsa_index_scores(q_idx, k_idx, w, seg=None, scores=None, ld: int | None = None, stream=None):
    """q_idx [B,S,Hi,Di] bf16, k_idx [B,S,Di] bf16, w [B,S,Hi] fp32/bf16, seg [B,S] int32.

    Returns scores fp32 [B,S,ld] (ld >= S, multiple of 4); only s <= t is written.
    """
    B, S, Hi, Di = q_idx.shape
    if ld is None:
        ld = (S + 3) // 4 * 4
    if scores is None:
        scores = torch.empty((B, S, ld), dtype=torch.float32, device=q_idx.device)
    ld = scores.shape[-1]
    w_dtype = DSA_F32 if w.dtype == torch.float32 else DSA_BF16
    rc = lib.dsa_index_scores(_dev(q_idx, "q_idx", torch.bfloat16), _dev(k_idx, "k_idx", torch.bfloat16),
                              _dev(w, "w"), w_dtype,
                              None if seg is None else _dev(seg, "seg", torch.int32),
                              B, S, Hi, Di, _dev(scores, "scores", torch.float32), ld,
                              _stream(stream))
    _check(rc, "dsa_index_scores")
    return scores


_FP8_DTYPES = (torch.uint8,) + ((torch.float8_e4m3fn,) if hasattr(torch, "float8_e4m3fn") else ())


def _dev8(t: torch.Tensor, name: str) -> int:
    if isinstance(t, torch.Tensor) and t.dtype not in _FP8_DTYPES:
        raise TypeError(f"{name} must hold e4m3 bytes (torch.uint8 or torch.float8_e4m3fn)")
    return _dev(t, name)


def dsa_index_scores_fp8(q_idx, k_idx, w, seg=None, k_scale=None, scores=None,
                         ld: int | None = None, stream=None):
    """q_idx [B,S,Hi,Di], k_idx [B,S,Di] as e4m3 bytes; k_scale fp32 [B,S] (> 0) or None.

    Returns scores fp32 [B,S,ld]: k_scale[s] * sum_h w * relu(q . k); only s <= t is written.
    """
    B, S, Hi, Di = q_idx.shape
    if ld is None:
        ld = (S + 3) // 4 * 4
    if scores is None:
        scores = torch.empty((B, S, ld), dtype=torch.float32, device=q_idx.device)
    ld = scores.shape[-1]
    w_dtype = DSA_F32 if w.dtype == torch.float32 else DSA_BF16
    rc = lib.dsa_index_scores_fp8(_dev8(q_idx, "q_idx"), _dev8(k_idx, "k_idx"),
                                  None if k_scale is None else _dev(k_scale, "k_scale", torch.float32),
                                  _dev(w, "w"), w_dtype,
                                  None if seg is None else _dev(seg, "seg", torch.int32),
                                  B, S, Hi, Di, _dev(scores, "scores", torch.float32), ld,
                                  _stream(stream))
    _check(rc, "dsa_index_scores_fp8")
    return scores


def _vals_out(vals, B, S, k, dev):
    """vals: None (not wanted), True (allocate) or an fp32 [B, S, k] tensor."""
    if vals is None or vals is False:
        return None
    if vals is True:
        return torch.empty((B, S, k), dtype=torch.float32, device=dev)
    return vals


def dsa_topk(scores, k: int, seg=None, S: int | None = None, idx=None, count=None, vals=None,
             stream=None):
    """scores fp32 [B,S,ld] -> (idx int32 [B,S,k] ascending / -1 padded, count int32 [B,S]).

    vals: True or an fp32 [B,S,k] tensor to have each slot's score as well (-inf at empty
    slots); the result is then (idx, count, vals).
    """
    B, S_, ld = scores.shape
    S = S_ if S is None else S
    if idx is None:
        idx = torch.empty((B, S, k), dtype=torch.int32, device=scores.device)
    if count is None:
        count = torch.empty((B, S), dtype=torch.int32, device=scores.device)
    vals = _vals_out(vals, B, S, k, scores.device)
    rc = lib.dsa_topk(_dev(scores, "scores", torch.float32), ld,
                      None if seg is None else _dev(seg, "seg", torch.int32), B, S, k,
                      _dev(idx, "idx", torch.int32), _dev(count, "count", torch.int32),
                      None if vals is None else _dev(vals, "vals", torch.float32), None, 0,
                      _stream(stream))
    _check(rc, "dsa_topk")
    return (idx, count) if vals is None else (idx, count, vals)


def fwd_workspace_bytes(B, S, H, Hkv, Dqk, Dv) -> int:
    return int(lib.dsa_sparse_attn_fwd_workspace_size(B, S, H, Hkv, Dqk, Dv))


def dsa_sparse_attn_fwd(Q, K, V, idx, scale: float, O=None, lse=None, ws=None, stream=None,
                        _entry: str = "dsa_sparse_attn_fwd"):
    """Q [B,S,H,Dqk], K [B,S,Hkv,Dqk], V [B,S,Hkv,Dv] bf16, idx [B,S,k] -> (O bf16, lse fp32).

    ws: a device byte buffer of at least fwd_workspace_bytes(...) (allocated here if None).
    """
    B, S, H, Dqk = Q.shape
    Hkv, Dv = V.shape[2], V.shape[3]
    k = idx.shape[2]
    if O is None:
        O = torch.empty((B, S, H, Dv), dtype=torch.bfloat16, device=Q.device)
    if lse is None:
        lse = torch.empty((B, S, H), dtype=torch.float32, device=Q.device)
    need = fwd_workspace_bytes(B, S, H, Hkv, Dqk, Dv)
    if ws is None and need > 0:
        ws = torch.empty((need,), dtype=torch.uint8, device=Q.device)
    rc = getattr(lib, _entry)(_dev(Q, "Q", torch.bfloat16), _dev(K, "K", torch.bfloat16),
                              _dev(V, "V", torch.bfloat16), _dev(idx, "idx", torch.int32),
                              B, S, H, Hkv, Dqk, Dv, k, float(scale),
                              _dev(O, "O", torch.bfloat16), _dev(lse, "lse", torch.float32),
                              None if ws is None else _dev(ws, "ws"),
                              0 if ws is None else ws.numel() * ws.element_size(),
                              _stream(stream))
    _check(rc, _entry)
    return O, lse


DSA_FWD_GATHER_TC, DSA_FWD_DENSE_TC, DSA_FWD_MMA_SYNC = 0, 1, 2


def dsa_sparse_attn_fwd_kernel(B, S, H, Hkv, Dqk, Dv, k, scale: float) -> int:
    """Which kernel dsa_sparse_attn_fwd runs for this shape (DSA_FWD_*; launches nothing)."""
    r = lib.dsa_sparse_attn_fwd_kernel(B, S, H, Hkv, Dqk, Dv, k, float(scale))
    if r < 0:
        raise DsaError(-r, "dsa_sparse_attn_fwd_kernel")
    return r


def dsa_sparse_attn_fwd_dense(Q, K, V, idx, scale: float, O=None, lse=None, ws=None,
                              stream=None):
    """dsa_sparse_attn_fwd through the dense-tile kernel only (same arguments and result)."""
    return dsa_sparse_attn_fwd(Q, K, V, idx, scale, O=O, lse=lse, ws=ws, stream=stream,
                               _entry="dsa_sparse_attn_fwd_dense")


def bwd_workspace_bytes(B, S, H, Hkv, Dqk, Dv) -> int:
    return int(lib.dsa_sparse_attn_bwd_workspace_size(B, S, H, Hkv, Dqk, Dv))


def dsa_sparse_attn_bwd(Q, K, V, idx, O, lse, dO, scale: float, dQ=None, dK=None, dV=None,
                        ws=None, stream=None, _entry: str = "dsa_sparse_attn_bwd"):
    """Gradients of the sparse attention -> (dQ [B,S,H,Dqk], dK [B,S,Hkv,Dqk], dV [B,S,Hkv,Dv])."""
    B, S, H, Dqk = Q.shape
    Hkv, Dv = V.shape[2], V.shape[3]
    k = idx.shape[2]
    dev = Q.device
    if dQ is None:
        dQ = torch.empty_like(Q)
    if dK is None:
        dK = torch.empty((B, S, Hkv, Dqk), dtype=torch.bfloat16, device=dev)
    if dV is None:
        dV = torch.empty((B, S, Hkv, Dv), dtype=torch.bfloat16, device=dev)
    need = bwd_workspace_bytes(B, S, H, Hkv, Dqk, Dv)
    if ws is None:   # the fp32 dK / dV accumulators and the dense-tile kernels' scratch
        ws = torch.empty((max(need, 16),), dtype=torch.uint8, device=dev)
    rc = getattr(lib, _entry)(_dev(Q, "Q", torch.bfloat16), _dev(K, "K", torch.bfloat16),
                              _dev(V, "V", torch.bfloat16), _dev(idx, "idx", torch.int32),
                              _dev(O, "O", torch.bfloat16), _dev(lse, "lse", torch.float32),
                              _dev(dO, "dO", torch.bfloat16), B, S, H, Hkv, Dqk, Dv, k,
                              float(scale), _dev(dQ, "dQ", torch.bfloat16),
                              _dev(dK, "dK", torch.bfloat16), _dev(dV, "dV", torch.bfloat16),
                              _dev(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, _entry)
    return dQ, dK, dV


def dsa_sparse_attn_bwd_dense(Q, K, V, idx, O, lse, dO, scale: float, dQ=None, dK=None,
                              dV=None, ws=None, stream=None):
    """dsa_sparse_attn_bwd through the dense-tile kernels only (same arguments and result)."""
    return dsa_sparse_attn_bwd(Q, K, V, idx, O, lse, dO, scale, dQ=dQ, dK=dK, dV=dV, ws=ws,
                               stream=stream, _entry="dsa_sparse_attn_bwd_dense")


DSA_BWD_GATHER_TC, DSA_BWD_DENSE_TC, DSA_BWD_MMA_SYNC = 0, 1, 2


def dsa_sparse_attn_bwd_kernel(B, S, H, Hkv, Dqk, Dv, k, scale: float) -> int:
    """Which kernels dsa_sparse_attn_bwd runs for this shape (DSA_BWD_*; launches nothing)."""
    r = lib.dsa_sparse_attn_bwd_kernel(B, S, H, Hkv, Dqk, Dv, k, float(scale))
    if r < 0:
        raise DsaError(-r, "dsa_sparse_attn_bwd_kernel")
    return r


def dsa_sparse_attn_bwd_noalloc(Q, K, V, idx, O, lse, dO, scale: float, dQ=None, dK=None,
                                dV=None, stream=None):
    """dsa_sparse_attn_bwd without a caller workspace: the library's fixed
    accumulator is used (see include/dsa.h for its size limit)."""
    B, S, H, Dqk = Q.shape
    Hkv, Dv = V.shape[2], V.shape[3]
    k = idx.shape[2]
    dev = Q.device
    if dQ is None:
        dQ = torch.empty_like(Q)
    if dK is None:
        dK = torch.empty((B, S, Hkv, Dqk), dtype=torch.bfloat16, device=dev)
    if dV is None:
        dV = torch.empty((B, S, Hkv, Dv), dtype=torch.bfloat16, device=dev)
    rc = lib.dsa_sparse_attn_bwd_noalloc(
        _dev(Q, "Q", torch.bfloat16), _dev(K, "K", torch.bfloat16), _dev(V, "V", torch.bfloat16),
        _dev(idx, "idx", torch.int32), _dev(O, "O", torch.bfloat16),
        _dev(lse, "lse", torch.float32), _dev(dO, "dO", torch.bfloat16), B, S, H, Hkv, Dqk, Dv, k,
        float(scale), _dev(dQ, "dQ", torch.bfloat16), _dev(dK, "dK", torch.bfloat16),
        _dev(dV, "dV", torch.bfloat16), _stream(stream))
    _check(rc, "dsa_sparse_attn_bwd_noalloc")
    return dQ, dK, dV


class HostPipeline:
    """Whole-layer steps from pinned host tensors to pinned host tensors.

    Host->device copies, the four stages and device->host copies run on three streams
    ordered by events, so that the copies overlap the kernels: the indexer starts as
    soon as its own (small) inputs have landed while Q, K, V, dO are still on their way,
    and the index lists and O leave while the backward runs. Consecutive steps overlap
    too: a step's indexer inputs load once the previous step's indexer has read them,
    and Q, K, V, dO are double-buffered, so the next step's load into the other set
    runs during this step's attention. Device buffers are allocated once; every stage
    runs in the library's kernels.
    """

    def __init__(self, B, S, Hi, Di, H, Dqk, Dv, topk, scale, backward=True, segments=False,
                 device=None, Hkv=1, indexer_loss=False, grad_scale=None, indexer_dtype="bf16",
                 fused_block_rows=0, stream_form=False):
        """indexer_loss: also run the indexer loss (objective grad_scale * sum of the
        per-query losses, default 1/(B*S)) and its gradient each step, returning kl,
        dq_idx, dk_idx and dw; the top-k hands the loss its selected scores slot by slot, so
        it runs with every form of the top-k. indexer_dtype "e4m3": q_idx / k_idx are e4m3
        bytes and the fp8 indexer runs. fused_block_rows > 0: the indexer and the top-k run
        fused through blocks of that many query rows (dsa_index_topk), with no [B, S, S]
        score matrix; with stream_form, in the streaming form (dsa_index_topk_stream: no
        score rows; the blocks are those its fallback redoes)."""
        if indexer_dtype not in ("bf16", "e4m3"):
            raise ValueError("indexer_dtype is 'bf16' or 'e4m3'")
        if indexer_loss and indexer_dtype != "bf16":
            raise ValueError("the indexer loss's backward reads the bf16 indexer inputs")
        dev = torch.device("cuda") if device is None else torch.device(device)
        self.dev, self.topk, self.scale, self.backward = dev, topk, scale, backward
        self.loss = indexer_loss
        self.fp8 = indexer_dtype == "e4m3"
        self.block_rows = fused_block_rows
        self.stream_form = bool(stream_form and fused_block_rows)
        self.grad_scale = 1.0 / (B * S) if grad_scale is None else grad_scale
        e = lambda *shape, dt=torch.bfloat16: torch.empty(shape, dtype=dt, device=dev)  # noqa: E731
        idt = torch.uint8 if self.fp8 else torch.bfloat16
        self.d = {"q_idx": e(B, S, Hi, Di, dt=idt), "k_idx": e(B, S, Di, dt=idt),
                  "w": e(B, S, Hi, dt=torch.float32)}
        if segments:
            self.d["seg"] = e(B, S, dt=torch.int32)
        self.big = []
        for _ in range(2):
            sets = {"Q": e(B, S, H, Dqk), "K": e(B, S, Hkv, Dqk), "V": e(B, S, Hkv, Dv)}
            if backward:
                sets["dO"] = e(B, S, H, Dv)
            self.big.append(sets)
        self.n = 0
        ld = (S + 3) // 4 * 4
        if fused_block_rows:   # one block of query rows of scores
            self.scores = None
            wsb = (index_topk_stream_workspace_bytes(B, S, fused_block_rows) if self.stream_form
                   else index_topk_workspace_bytes(B, S, fused_block_rows))
            self.topk_ws = e(max(wsb, 16), dt=torch.uint8)
        else:
            self.scores = e(B, S, ld, dt=torch.float32)
        self.fwd_ws = e(max(fwd_workspace_bytes(B, S, H, Hkv, Dqk, Dv), 16), dt=torch.uint8)
        self.out = {"idx": e(B, S, topk, dt=torch.int32), "count": e(B, S, dt=torch.int32),
                    "O": e(B, S, H, Dv), "lse": e(B, S, H, dt=torch.float32)}
        if backward:
            self.out.update({"dQ": e(B, S, H, Dqk), "dK": e(B, S, Hkv, Dqk),
                             "dV": e(B, S, Hkv, Dv)})
            self.ws = e(bwd_workspace_bytes(B, S, H, Hkv, Dqk, Dv), dt=torch.uint8)
        self.sel = None
        if indexer_loss:
            f32 = torch.float32
            self.dI = e(B, S, topk, dt=f32)
            self.sel = e(B, S, topk, dt=f32)   # the selected scores, by slot
            self.out.update({"kl": e(B, S, dt=f32), "dq_idx": e(B, S, Hi, Di, dt=f32),
                             "dk_idx": e(B, S, Di, dt=f32), "dw": e(B, S, Hi, dt=f32)})
        self.s_in, self.s_c, self.s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
        ev = lambda: torch.cuda.Event()  # noqa: E731
        # events of earlier steps that the next one must respect
        self.ev_idx_read = None
        self.ev_attn_read = [None, None]   # per Q/K/V/dO set: its last reader is done
        self.ev_out1 = self.ev_out2 = self.ev_out3 = self.ev_out4 = None
        self._ev = ev

    def _wait(self, stream, event):
        if event is not None:
            stream.wait_event(event)

    @staticmethod
    def _bits(dst, src):
        """dst viewed with src's dtype when only the element type name differs
        (bf16 data held as 16-bit integers on the host): a bit copy."""
        return dst if dst.dtype == src.dtype else dst.view(src.dtype)

    def step(self, h_in: dict, h_out: dict):
        """Enqueue one step: h_in / h_out hold pinned host tensors named like the
        device buffers (inputs q_idx, k_idx, w, [seg], Q, K, V, [dO]; outputs idx,
        count, O, lse, [dQ, dK, dV], [kl, dq_idx, dk_idx, dw]). Returns the event that
        completes the step."""
        d, o, ev = self.d, self.out, self._ev
        par = self.n & 1
        bd = self.big[par]
        small = [n for n in ("q_idx", "k_idx", "w", "seg") if n in d]
        big = [n for n in ("Q", "K", "V", "dO") if n in bd]
        # host -> device
        with torch.cuda.stream(self.s_in):
            self._wait(self.s_in, self.ev_idx_read)
            for n in small:
                self._bits(d[n], h_in[n]).copy_(h_in[n], non_blocking=True)
            in1 = ev()
            in1.record(self.s_in)
            self._wait(self.s_in, self.ev_attn_read[par])
            for n in big:
                self._bits(bd[n], h_in[n]).copy_(h_in[n], non_blocking=True)
            in2 = ev()
            in2.record(self.s_in)
        # the layer
        sc = self.s_c
        sc.wait_event(in1)
        self._wait(sc, self.ev_out1)
        if self.block_rows:
            fuse = dsa_index_topk_stream if self.stream_form else dsa_index_topk
            fuse(d["q_idx"], d["k_idx"], d["w"], self.topk, d.get("seg"),
                 block_rows=self.block_rows, idx=o["idx"], count=o["count"], ws=self.topk_ws,
                 stream=sc, vals=self.sel)
        elif self.fp8:
            dsa_index_scores_fp8(d["q_idx"], d["k_idx"], d["w"], d.get("seg"),
                                 scores=self.scores, stream=sc)
        else:
            dsa_index_scores(d["q_idx"], d["k_idx"], d["w"], d.get("seg"), scores=self.scores,
                             stream=sc)
        idx_read = ev()
        idx_read.record(sc)
        if not self.block_rows:
            dsa_topk(self.scores, self.topk, d.get("seg"), idx=o["idx"], count=o["count"],
                     vals=self.sel, stream=sc)
        topk_done = ev()
        topk_done.record(sc)
        sc.wait_event(in2)
        self._wait(sc, self.ev_out2)
        dsa_sparse_attn_fwd(bd["Q"], bd["K"], bd["V"], o["idx"], self.scale, O=o["O"],
                            lse=o["lse"], ws=self.fwd_ws, stream=sc)
        fwd_done = ev()
        fwd_done.record(sc)
        bwd_done = fwd_done
        if self.backward:
            self._wait(sc, self.ev_out3)
            dsa_sparse_attn_bwd(bd["Q"], bd["K"], bd["V"], o["idx"], o["O"], o["lse"], bd["dO"],
                                self.scale, dQ=o["dQ"], dK=o["dK"], dV=o["dV"], ws=self.ws,
                                stream=sc)
            bwd_done = ev()
            bwd_done.record(sc)
        attn_read = bwd_done
        if self.loss:
            # reads Q, K, the selected scores and the indexer inputs: the next step's copies
            # into them wait for it (idx_read, attn_read)
            self._wait(sc, self.ev_out4)
            dsa_indexer_loss(bd["Q"], bd["K"], o["idx"], o["lse"], None, self.scale,
                             self.grad_scale, kl=o["kl"], dI=self.dI, stream=sc,
                             sel_scores=self.sel)
            dsa_indexer_loss_bwd(d["q_idx"], d["k_idx"], d["w"], o["idx"], self.dI,
                                 dq_idx=o["dq_idx"], dk_idx=o["dk_idx"], dw=o["dw"], stream=sc)
            loss_done = ev()
            loss_done.record(sc)
            idx_read = attn_read = loss_done
        # device -> host
        with torch.cuda.stream(self.s_out):
            self.s_out.wait_event(topk_done)
            for n in ("idx", "count"):
                h_out[n].copy_(self._bits(o[n], h_out[n]), non_blocking=True)
            out1 = ev()
            out1.record(self.s_out)
            self.s_out.wait_event(fwd_done)
            for n in ("O", "lse"):
                h_out[n].copy_(self._bits(o[n], h_out[n]), non_blocking=True)
            out2 = ev()
            out2.record(self.s_out)
            out3 = out2
            if self.backward:
                self.s_out.wait_event(bwd_done)
                for n in ("dQ", "dK", "dV"):
                    h_out[n].copy_(self._bits(o[n], h_out[n]), non_blocking=True)
                out3 = ev()
                out3.record(self.s_out)
            out4 = out3
            if self.loss:
                self.s_out.wait_event(loss_done)
                for n in ("kl", "dq_idx", "dk_idx", "dw"):
                    h_out[n].copy_(o[n], non_blocking=True)
                out4 = ev()
                out4.record(self.s_out)
        self.ev_idx_read = idx_read
        self.ev_attn_read[par] = attn_read
        self.ev_out1, self.ev_out2, self.ev_out3, self.ev_out4 = out1, out2, out3, out4
        self.n += 1
        return out4


def index_topk_workspace_bytes(B, S, block_rows) -> int:
    return int(lib.dsa_index_topk_workspace_size(B, S, block_rows))


def index_topk_stream_workspace_bytes(B, S, block_rows) -> int:
    return int(lib.dsa_index_topk_stream_workspace_size(B, S, block_rows))


def dsa_index_topk_stream(q_idx, k_idx, w, k: int, seg=None, block_rows: int | None = None,
                          idx=None, count=None, ws=None, stream=None, k_scale=None, vals=None):
    """Indexer scores and top-k with no score rows in memory (the streaming form).

    Same arguments and results as dsa_index_topk (vals needs k <= 2048); `block_rows` (a
    multiple of 256, default S / 8 rounded up) sizes the blocks that the memory form redoes
    for rows the sampled window does not settle.
    """
    B, S, Hi, Di = q_idx.shape
    dev = q_idx.device
    if block_rows is None:
        block_rows = max(256, (S // 8 + 255) // 256 * 256)
    if idx is None:
        idx = torch.empty((B, S, k), dtype=torch.int32, device=dev)
    if count is None:
        count = torch.empty((B, S), dtype=torch.int32, device=dev)
    need = index_topk_stream_workspace_bytes(B, S, block_rows)
    if ws is None:
        ws = torch.empty((max(need, 16),), dtype=torch.uint8, device=dev)
    w_dtype = DSA_F32 if w.dtype == torch.float32 else DSA_BF16
    vals = _vals_out(vals, B, S, k, dev)
    tail = (None if seg is None else _dev(seg, "seg", torch.int32), B, S, Hi, Di, k, block_rows,
            _dev(idx, "idx", torch.int32), _dev(count, "count", torch.int32),
            None if vals is None else _dev(vals, "vals", torch.float32), _dev(ws, "ws"),
            ws.numel() * ws.element_size(), _stream(stream))
    if q_idx.dtype in _FP8_DTYPES:
        rc = lib.dsa_index_topk_stream_fp8(_dev8(q_idx, "q_idx"), _dev8(k_idx, "k_idx"),
                                           None if k_scale is None else _dev(k_scale, "k_scale",
                                                                             torch.float32),
                                           _dev(w, "w"), w_dtype, *tail)
        _check(rc, "dsa_index_topk_stream_fp8")
    else:
        rc = lib.dsa_index_topk_stream(_dev(q_idx, "q_idx", torch.bfloat16),
                                       _dev(k_idx, "k_idx", torch.bfloat16), _dev(w, "w"),
                                       w_dtype, *tail)
        _check(rc, "dsa_index_topk_stream")
    return (idx, count) if vals is None else (idx, count, vals)


def dsa_index_topk(q_idx, k_idx, w, k: int, seg=None, block_rows: int = 2048, idx=None,
                   count=None, ws=None, stream=None, k_scale=None, vals=None):
    """Indexer scores and top-k fused through blocks of query rows (no [B,S,S] scores).

    Same arguments and results as dsa_index_scores (or dsa_index_scores_fp8, for e4m3
    q_idx / k_idx, with k_scale) followed by dsa_topk (vals as there); the scores of one
    block of block_rows query rows (a multiple of 256) live in `ws`.
    """
    B, S, Hi, Di = q_idx.shape
    dev = q_idx.device
    if idx is None:
        idx = torch.empty((B, S, k), dtype=torch.int32, device=dev)
    if count is None:
        count = torch.empty((B, S), dtype=torch.int32, device=dev)
    need = index_topk_workspace_bytes(B, S, block_rows)
    if ws is None:
        ws = torch.empty((max(need, 16),), dtype=torch.uint8, device=dev)
    w_dtype = DSA_F32 if w.dtype == torch.float32 else DSA_BF16
    vals = _vals_out(vals, B, S, k, dev)
    tail = (None if seg is None else _dev(seg, "seg", torch.int32), B, S, Hi, Di, k, block_rows,
            _dev(idx, "idx", torch.int32), _dev(count, "count", torch.int32),
            None if vals is None else _dev(vals, "vals", torch.float32), _dev(ws, "ws"),
            ws.numel() * ws.element_size(), _stream(stream))
    if q_idx.dtype in _FP8_DTYPES:
        rc = lib.dsa_index_topk_fp8(_dev8(q_idx, "q_idx"), _dev8(k_idx, "k_idx"),
                                    None if k_scale is None else _dev(k_scale, "k_scale",
                                                                      torch.float32),
                                    _dev(w, "w"), w_dtype, *tail)
        _check(rc, "dsa_index_topk_fp8")
    else:
        rc = lib.dsa_index_topk(_dev(q_idx, "q_idx", torch.bfloat16),
                                _dev(k_idx, "k_idx", torch.bfloat16), _dev(w, "w"), w_dtype,
                                *tail)
        _check(rc, "dsa_index_topk")
    return (idx, count) if vals is None else (idx, count, vals)


def dsa_indexer_loss(Q, K, idx, lse, scores, scale: float, grad_scale: float = 1.0, kl=None,
                     dI=None, stream=None, sel_scores=None):
    """Indexer auxiliary loss -> (kl fp32 [B,S], dI fp32 [B,S,k]).

    Q [B,S,H,Dqk] bf16, K [B,S,1,Dqk] bf16, idx [B,S,k] int32, lse [B,S,H] fp32 (the
    attention forward's), scores [B,S,ld] fp32 (the index scores), or scores=None and
    sel_scores [B,S,k] fp32: the selected keys' scores by slot (the top-k's vals). dI is
    the gradient of grad_scale * kl.sum() with respect to the score at each slot of idx.
    """
    B, S, H, Dqk = Q.shape
    Hkv = K.shape[2]
    k = idx.shape[2]
    if kl is None:
        kl = torch.empty((B, S), dtype=torch.float32, device=Q.device)
    if dI is None:
        dI = torch.empty((B, S, k), dtype=torch.float32, device=Q.device)
    rc = lib.dsa_indexer_loss(_dev(Q, "Q", torch.bfloat16), _dev(K, "K", torch.bfloat16),
                              _dev(idx, "idx", torch.int32), _dev(lse, "lse", torch.float32),
                              _dev(scores if scores is not None else sel_scores, "scores",
                                   torch.float32),
                              scores.shape[-1] if scores is not None else 0, B, S, H,
                              Hkv, Dqk, k, float(scale), float(grad_scale),
                              _dev(kl, "kl", torch.float32), _dev(dI, "dI", torch.float32),
                              _stream(stream))
    _check(rc, "dsa_indexer_loss")
    return kl, dI


def dsa_indexer_loss_bwd(q_idx, k_idx, w, idx, dI, dq_idx=None, dk_idx=None, dw=None,
                         stream=None):
    """Gradient of the indexer loss into the indexer inputs -> (dq_idx, dk_idx, dw), fp32.

    q_idx [B,S,Hi,Di] bf16, k_idx [B,S,Di] bf16, w [B,S,Hi] fp32, idx [B,S,k] int32,
    dI [B,S,k] fp32 (from dsa_indexer_loss).
    """
    B, S, Hi, Di = q_idx.shape
    k = idx.shape[2]
    dev = q_idx.device
    if dq_idx is None:
        dq_idx = torch.empty((B, S, Hi, Di), dtype=torch.float32, device=dev)
    if dk_idx is None:
        dk_idx = torch.empty((B, S, Di), dtype=torch.float32, device=dev)
    if dw is None:
        dw = torch.empty((B, S, Hi), dtype=torch.float32, device=dev)
    rc = lib.dsa_indexer_loss_bwd(_dev(q_idx, "q_idx", torch.bfloat16),
                                  _dev(k_idx, "k_idx", torch.bfloat16), _dev(w, "w", torch.float32),
                                  _dev(idx, "idx", torch.int32), _dev(dI, "dI", torch.float32),
                                  B, S, Hi, Di, k, _dev(dq_idx, "dq_idx", torch.float32),
                                  _dev(dk_idx, "dk_idx", torch.float32), _dev(dw, "dw", torch.float32),
                                  _stream(stream))
    _check(rc, "dsa_indexer_loss_bwd")
    return dq_idx, dk_idx, dw


def dsa_layer(q_idx, k_idx, w, Q, K, V, topk: int, scale: float, seg=None, dO=None, stream=None):
    """The whole hot path: scores -> top-k -> sparse attention forward (and backward if dO)."""
    scores = dsa_index_scores(q_idx, k_idx, w, seg, stream=stream)
    idx, count = dsa_topk(scores, topk, seg, stream=stream)
    O, lse = dsa_sparse_attn_fwd(Q, K, V, idx, scale, stream=stream)
    out = {"scores": scores, "idx": idx, "count": count, "O": O, "lse": lse}
    if dO is not None:
        out["dQ"], out["dK"], out["dV"] = dsa_sparse_attn_bwd(Q, K, V, idx, O, lse, dO, scale,
                                                               stream=stream)
    return out
