"""Seeded synthetic inputs for the DSA layer workloads.

This package only draws random numbers (see ``synth.c``); it holds none of the
indexer / top-k / attention arithmetic. The fp64 oracle and the CUDA path are
both fed from it, so they see identical inputs.

Workload shapes follow the DeepSeek-V3.2 indexer configuration (64 indexer
heads x 128 dims, index_topk 2048: "DeepSeek3.2: Onboard sparse attention",
section "2. Onboard deepseek3.2-671b config") and the MLA head dims
(qk 192 = 128 nope + 64 rope, v 128). Indexer inputs are small dyadic values so
that every fp32 indexer sum is exact; attention inputs are N(0,1) rounded to
bf16. The unaligned S=489 case follows "Add Flash Attention Support to
Deepseek v4" (non-power-of-two sequence lengths).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

# stream ids: one independent counter stream per tensor
STREAM_Q_IDX, STREAM_K_IDX, STREAM_W = 1, 2, 3
STREAM_Q, STREAM_K, STREAM_V, STREAM_DO = 4, 5, 6, 7
STREAM_SEG = 8
STREAM_K_SCALE = 9
STREAM_ROWS = 64


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``libsynth.so`` next to it (gcc, -O2)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-o", tmp,
                    _SRC, "-lm", "-lpthread"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, u64, ci, vp = ctypes.c_int64, ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p
            lib.synth_normal_bf16.argtypes = [vp, i64, u64, u64, ci]
            lib.synth_dyadic_bf16.argtypes = [vp, i64, u64, u64, i64, i64, ci, ci]
            lib.synth_dyadic_f32.argtypes = [vp, i64, u64, u64, i64, i64, ci, ci]
            lib.synth_signed_nonzero_f32.argtypes = [vp, i64, u64, u64, i64, ci, ci]
            lib.synth_segments.argtypes = [vp, ci, ci, ci, u64, u64]
            lib.synth_segments.restype = ci
            lib.synth_word.argtypes = [u64, u64, u64]
            lib.synth_word.restype = u64
            _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal_bf16(shape, seed: int, stream: int) -> np.ndarray:
    """N(0,1) values rounded to bf16; returned as uint16 bit patterns."""
    out = np.empty(shape, dtype=np.uint16)
    _load().synth_normal_bf16(out.ctypes.data, out.size, seed, stream, _threads())
    return out


def dyadic_bf16(shape, seed: int, stream: int, lo: int, hi: int, denom_log2: int) -> np.ndarray:
    """i / 2**denom_log2, i uniform on [lo, hi]; uint16 bf16 bit patterns."""
    out = np.empty(shape, dtype=np.uint16)
    _load().synth_dyadic_bf16(out.ctypes.data, out.size, seed, stream, lo, hi, denom_log2, _threads())
    return out


def dyadic_f32(shape, seed: int, stream: int, lo: int, hi: int, denom_log2: int) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _load().synth_dyadic_f32(out.ctypes.data, out.size, seed, stream, lo, hi, denom_log2, _threads())
    return out


def signed_nonzero_f32(shape, seed: int, stream: int, hi: int, denom_log2: int) -> np.ndarray:
    """i / 2**denom_log2, i uniform on {-hi..-1, 1..hi}."""
    out = np.empty(shape, dtype=np.float32)
    _load().synth_signed_nonzero_f32(out.ctypes.data, out.size, seed, stream, hi, denom_log2, _threads())
    return out


def segments(B: int, S: int, ndocs: int, seed: int, stream: int = STREAM_SEG) -> np.ndarray:
    """Segment ids [B, S] int32: ndocs contiguous documents per row."""
    out = np.empty((B, S), dtype=np.int32)
    rc = _load().synth_segments(out.ctypes.data, B, S, ndocs, seed, stream)
    if rc != 0:
        raise ValueError("bad segment request")
    return out


def words(seed: int, stream: int, n: int) -> np.ndarray:
    lib = _load()
    return np.array([lib.synth_word(seed, stream, i) for i in range(n)], dtype=np.uint64)


def bf16_to_f32(u16: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (u16.astype(np.uint32) << 16).view(np.float32)


def e4m3_bytes(values) -> np.ndarray:
    """Exact OCP FP8 E4M3 bytes (uint8) of values that e4m3 represents exactly.

    The conversion is torch's float8_e4m3fn cast; values that would round raise.
    """
    import torch
    v = torch.from_numpy(np.ascontiguousarray(values, dtype=np.float32))
    f8 = v.to(torch.float8_e4m3fn)
    if not torch.equal(f8.to(torch.float32), v):
        raise ValueError("value not exactly representable in e4m3")
    return f8.view(torch.uint8).numpy().copy()


def pow2_scales(shape, seed: int, stream: int, lo: int, hi: int) -> np.ndarray:
    """2**j with j uniform on the integers lo..hi, float32."""
    j = dyadic_f32(shape, seed, stream, lo, hi, 0)
    return np.exp2(j).astype(np.float32)


@dataclass(frozen=True)
class Workload:
    """Shapes and input distributions of one synthetic DSA layer workload."""
    name: str
    seed: int
    B: int
    S: int
    Hi: int
    Di: int
    topk: int
    H: int
    Dqk: int
    Dv: int
    backward: bool
    ndocs: int = 0          # 0: no segment ids (plain causal)
    Hkv: int = 1
    idx_int_range: tuple = (-8, 8)   # q_idx / k_idx = i / 2**idx_denom_log2
    idx_denom_log2: int = 3
    w_kind: str = "dyadic"           # "dyadic": j / 2**w_denom_log2, j on w_range
    w_range: tuple = (-1, 1)         # "signed_nonzero": {+-1..+-w_range[1]} / 2**w_denom_log2
    w_denom_log2: int = 4
    description: str = field(default="", compare=False)

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.Dqk))

    @property
    def tokens(self) -> int:
        return self.B * self.S

    def replace(self, **kw) -> "Workload":
        d = {f: getattr(self, f) for f in self.__dataclass_fields__}
        d.update(kw)
        return Workload(**d)


WORKLOADS = {
    "tiny_s128": Workload(
        "tiny_s128", seed=0, B=1, S=128, Hi=4, Di=32, topk=4, H=2, Dqk=32, Dv=32, backward=True,
        idx_int_range=(-4, 4), idx_denom_log2=0, w_kind="signed_nonzero", w_range=(1, 8),
        w_denom_log2=3,
        description="tiny DSA layer: 4 idx heads x 32, top-4, 2 heads x 32/32, fwd+bwd"),
    "small2b_s4096": Workload(
        "small2b_s4096", seed=1, B=2, S=4096, Hi=64, Di=128, topk=2048, H=16, Dqk=192, Dv=128,
        backward=False,
        description="2B-scale DSA layer: 64 idx heads x 128, top-2048, 16 heads, fwd"),
    "v32_671b_s16k": Workload(
        "v32_671b_s16k", seed=2, B=1, S=16384, Hi=64, Di=128, topk=2048, H=128, Dqk=192, Dv=128,
        backward=True,
        description="DS-v3.2-671B layer shape: 64 idx heads x 128, top-2048, 128 heads, fwd+bwd"),
    "v32_671b_s4096": Workload(
        "v32_671b_s4096", seed=2, B=1, S=4096, Hi=64, Di=128, topk=2048, H=128, Dqk=192, Dv=128,
        backward=True,
        description="DS-v3.2-671B layer shape cut to S=4096 (profiling size), fwd+bwd"),
    "long_s128k": Workload(
        "long_s128k", seed=3, B=1, S=131072, Hi=64, Di=128, topk=2048, H=128, Dqk=192, Dv=128,
        backward=False,
        description="long-context DSA layer, S=131072, fwd"),
    "packed_s4096": Workload(
        "packed_s4096", seed=4, B=4, S=4096, Hi=64, Di=128, topk=512, H=16, Dqk=192, Dv=128,
        backward=True, ndocs=3,
        description="packed training step: 3 documents per row, top-512, 16 heads, fwd+bwd"),
    "mla_perhead_s4096": Workload(
        "mla_perhead_s4096", seed=5, B=1, S=4096, Hi=64, Di=128, topk=2048, H=128, Hkv=128,
        Dqk=192, Dv=128, backward=True,
        description="DS-v3.2 layer shape at S=4096 with per-head K/V (each of the 128 heads "
                    "has its own 192/128 K/V rows), top-2048, fwd+bwd"),
    "packed_s489": Workload(
        "packed_s489", seed=4, B=1, S=489, Hi=64, Di=128, topk=512, H=16, Dqk=192, Dv=128,
        backward=True, ndocs=3,
        description="unaligned packed case S=489, same dims"),
}


def indexer_inputs(wl: Workload) -> dict:
    """q_idx [B,S,Hi,Di] bf16, k_idx [B,S,Di] bf16, w [B,S,Hi] f32, seg [B,S] int32 or None."""
    lo, hi = wl.idx_int_range
    q = dyadic_bf16((wl.B, wl.S, wl.Hi, wl.Di), wl.seed, STREAM_Q_IDX, lo, hi, wl.idx_denom_log2)
    k = dyadic_bf16((wl.B, wl.S, wl.Di), wl.seed, STREAM_K_IDX, lo, hi, wl.idx_denom_log2)
    if wl.w_kind == "dyadic":
        w = dyadic_f32((wl.B, wl.S, wl.Hi), wl.seed, STREAM_W, wl.w_range[0], wl.w_range[1],
                       wl.w_denom_log2)
    else:
        w = signed_nonzero_f32((wl.B, wl.S, wl.Hi), wl.seed, STREAM_W, wl.w_range[1],
                               wl.w_denom_log2)
    seg = segments(wl.B, wl.S, wl.ndocs, wl.seed) if wl.ndocs else None
    return {"q_idx": q, "k_idx": k, "w": w, "seg": seg}


def indexer_inputs_fp8(wl: Workload, k_scale: str = "none") -> dict:
    """indexer_inputs with q_idx / k_idx as e4m3 bytes (the same dyadic values) and a per-key
    scale: "none" (None), "pow2" (2**j, j in -2..2) or "dyadic" (i/64, i in 33..127)."""
    inp = indexer_inputs(wl)
    inp["q_idx"] = e4m3_bytes(bf16_to_f32(inp["q_idx"]))
    inp["k_idx"] = e4m3_bytes(bf16_to_f32(inp["k_idx"]))
    if k_scale == "none":
        inp["k_scale"] = None
    elif k_scale == "pow2":
        inp["k_scale"] = pow2_scales((wl.B, wl.S), wl.seed, STREAM_K_SCALE, -2, 2)
    else:
        inp["k_scale"] = dyadic_f32((wl.B, wl.S), wl.seed, STREAM_K_SCALE, 33, 127, 6)
    return inp


def attention_inputs(wl: Workload, with_grad: bool | None = None) -> dict:
    """Q [B,S,H,Dqk], K [B,S,Hkv,Dqk], V [B,S,Hkv,Dv], dO [B,S,H,Dv]; bf16 bit patterns."""
    with_grad = wl.backward if with_grad is None else with_grad
    out = {
        "Q": normal_bf16((wl.B, wl.S, wl.H, wl.Dqk), wl.seed, STREAM_Q),
        "K": normal_bf16((wl.B, wl.S, wl.Hkv, wl.Dqk), wl.seed, STREAM_K),
        "V": normal_bf16((wl.B, wl.S, wl.Hkv, wl.Dv), wl.seed, STREAM_V),
    }
    if with_grad:
        out["dO"] = normal_bf16((wl.B, wl.S, wl.H, wl.Dv), wl.seed, STREAM_DO)
    return out


def sample_rows(wl: Workload, n_uniform: int, seed_offset: int = 0) -> np.ndarray:
    """Flat query rows b*S + t: t in {0, k-1, k, S-1} plus n_uniform uniform draws, per batch."""
    rows = []
    for b in range(wl.B):
        ts = {0, min(wl.topk - 1, wl.S - 1), min(wl.topk, wl.S - 1), wl.S - 1}
        lib = _load()
        for i in range(n_uniform):
            wv = lib.synth_word(wl.seed + seed_offset, STREAM_ROWS + b, i)
            ts.add(int(((wv >> 32) * wl.S) >> 32))
        rows.extend(b * wl.S + t for t in sorted(ts))
    return np.array(rows, dtype=np.int64)
