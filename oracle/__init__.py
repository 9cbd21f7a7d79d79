"""fp64 CPU oracle for the Inkling attention block (sconv K/V + relative-bias GQA).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's CPU
baseline leg are the only callers.  The library's product path never imports this
package, and this package imports nothing from the library.

`oracle.c` holds the definitions (sconv with its cache, paged relative-bias attention);
this module compiles it with gcc on first use and marshals numpy/torch CPU arrays.
`brute.py` is a second, pure-Python statement of the same attention used to pin the C
code on tiny inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lib = None

STATUS = {0: "ok", 1: "invalid argument", 2: "block id out of range", 3: "out of memory"}


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so (plain C, gcc, -O2, pthreads)."""
    src = os.path.join(_HERE, "oracle.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src):
        return _SO
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _SO + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared",
                           "-pthread", "-o", tmp, src, "-lm"])
    os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P = ctypes.c_void_p
        L.oracle_bf16_round.restype = ctypes.c_uint16
        L.oracle_bf16_round.argtypes = [ctypes.c_double]
        L.oracle_bf16_to_double.restype = ctypes.c_double
        L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_sconv_kv.restype = ctypes.c_int
        L.oracle_sconv_kv.argtypes = [P, P, P, P, P, P, P, P, P, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int64]
        L.oracle_sconv_dense.restype = ctypes.c_int
        L.oracle_sconv_dense.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        L.oracle_sconv_rollback.restype = ctypes.c_int
        L.oracle_sconv_rollback.argtypes = [P, P, P, P, P, P, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int]
        L.oracle_e4m3_round.restype = ctypes.c_uint8
        L.oracle_e4m3_round.argtypes = [ctypes.c_double]
        L.oracle_e4m3_to_double.restype = ctypes.c_double
        L.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        L.oracle_sconv_kv_fp8.restype = ctypes.c_int
        L.oracle_sconv_kv_fp8.argtypes = [P, P, P, P, P, P, P, P, P, ctypes.c_double,
                                          ctypes.c_double, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int64]
        L.oracle_rel_attn_fp8.restype = ctypes.c_int
        L.oracle_rel_attn_fp8.argtypes = [P, P, P, ctypes.c_double, ctypes.c_double, P,
                                          ctypes.c_int, P, P, P, ctypes.c_int, ctypes.c_double,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int64, P, ctypes.c_int, P, P,
                                          ctypes.c_int]
        L.oracle_rel_attn.restype = ctypes.c_int
        L.oracle_rel_attn.argtypes = [P, P, P, P, ctypes.c_int, P, P, P, ctypes.c_int,
                                      ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int64, P, ctypes.c_int,
                                      P, P, ctypes.c_int]
        _lib = L
    return _lib


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _u16(t) -> np.ndarray:
    """A C-contiguous uint16 numpy view of a bf16 CPU tensor (or pass a uint16 array)."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    assert t.dtype == torch.bfloat16 and t.device.type == "cpu"
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _arr(t, dtype) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        assert t.device.type == "cpu"
        t = t.contiguous().numpy()
    return np.ascontiguousarray(t, dtype=dtype)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def bf16_round(y: float) -> int:
    """Round a float64 to bf16 (nearest, ties to even) in one step; returns the bits."""
    return int(lib().oracle_bf16_round(float(y)))


def bf16_bits_to_float(b: int) -> float:
    return float(lib().oracle_bf16_to_double(int(b) & 0xFFFF))


def sconv_kv(k_raw, v_raw, w_k, w_v, state, cu_q_lens, slot_mapping, k_cache, v_cache):
    """Sconv on K and V of the new tokens into the paged caches, and the state update.

    All arguments are CPU tensors (bf16 / fp32 / int32 / int64).  `state`, `k_cache` and
    `v_cache` are updated in place (they must be contiguous bf16 CPU tensors)."""
    for t in (state, k_cache, v_cache):
        assert t.is_contiguous() and t.dtype == torch.bfloat16 and t.device.type == "cpu"
    kr, vr = _u16(k_raw), _u16(v_raw)
    wk, wv = _arr(w_k, np.float32), _arr(w_v, np.float32)
    st = state.view(torch.int16).numpy().view(np.uint16)
    kc = k_cache.view(torch.int16).numpy().view(np.uint16)
    vc = v_cache.view(torch.int16).numpy().view(np.uint16)
    cu = _arr(cu_q_lens, np.int32)
    sm = _arr(slot_mapping, np.int64)
    B = cu.shape[0] - 1
    T = kr.shape[0] if kr.ndim == 2 else 0
    hkv = kc.shape[1]
    rc = lib().oracle_sconv_kv(_ptr(kr), _ptr(vr), _ptr(wk), _ptr(wv), _ptr(st), _ptr(cu),
                               _ptr(sm), _ptr(kc), _ptr(vc), B, T, hkv, kc.shape[0])
    if rc != 0:
        raise RuntimeError(f"oracle_sconv_kv: {STATUS.get(rc, rc)}")


def rel_attn(q, k_cache, v_cache, block_table, cu_q_lens, seq_lens, bias, *, scale: float,
             window: int, rows: Optional[Sequence[int]] = None, n_threads: Optional[int] = None):
    """Relative-bias GQA attention for the query tokens `rows` (default: all), all heads.

    Returns (out [n_rows, Hq, 128] float64, lse [n_rows, Hq] float64, natural log)."""
    qa = _u16(q)
    kc, vc = _u16(k_cache), _u16(v_cache)
    bt = _arr(block_table, np.int32)
    cu = _arr(cu_q_lens, np.int32)
    sl = _arr(seq_lens, np.int32)
    bi = _arr(bias, np.float32)
    T, hq = qa.shape[0], qa.shape[1]
    hkv = kc.shape[1]
    rows = np.arange(T, dtype=np.int32) if rows is None else _arr(rows, np.int32)
    out = np.zeros((rows.shape[0], hq, 128), dtype=np.float64)
    lse = np.zeros((rows.shape[0], hq), dtype=np.float64)
    rc = lib().oracle_rel_attn(_ptr(qa), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(cu),
                               _ptr(sl), _ptr(bi), bi.shape[1], float(scale), int(window),
                               cu.shape[0] - 1, T, hq, hkv, kc.shape[0], _ptr(rows),
                               rows.shape[0], _ptr(out), _ptr(lse),
                               host_cores() if n_threads is None else int(n_threads))
    if rc != 0:
        raise RuntimeError(f"oracle_rel_attn: {STATUS.get(rc, rc)}")
    return out, lse


def sconv_dense(x, w, state, cu_q_lens):
    """Sconv on one dense stream: returns y [T, C] bf16; `state` [B, 3, C] updated in place."""
    assert state.is_contiguous() and state.dtype == torch.bfloat16 and state.device.type == "cpu"
    xa = _u16(x)
    wa = _arr(w, np.float32)
    st = state.view(torch.int16).numpy().view(np.uint16)
    cu = _arr(cu_q_lens, np.int32)
    T, C = xa.shape
    y = torch.empty((T, C), dtype=torch.bfloat16)
    ya = y.view(torch.int16).numpy().view(np.uint16)
    rc = lib().oracle_sconv_dense(_ptr(xa), _ptr(wa), _ptr(st), _ptr(cu), _ptr(ya),
                                  cu.shape[0] - 1, T, C)
    if rc != 0:
        raise RuntimeError(f"oracle_sconv_dense: {STATUS.get(rc, rc)}")
    return y


def sconv_rollback(state_before, x0, x1, cu_q_lens, accepted):
    """Sconv state after keeping only the first accepted[b] new tokens of a step.

    streams = 2 when x1 is given (K/V pair state [B, 2, 3, C]), else 1 ([B, 3, C])."""
    sb = _u16(state_before)
    a0 = _u16(x0)
    a1 = _u16(x1) if x1 is not None else a0
    cu = _arr(cu_q_lens, np.int32)
    acc = _arr(accepted, np.int32)
    streams = 2 if x1 is not None else 1
    C = a0.shape[1]
    out = torch.empty(tuple(state_before.shape), dtype=torch.bfloat16)
    oa = out.view(torch.int16).numpy().view(np.uint16)
    rc = lib().oracle_sconv_rollback(_ptr(sb), _ptr(a0), _ptr(a1), _ptr(cu), _ptr(acc),
                                     _ptr(oa), cu.shape[0] - 1, C, streams)
    if rc != 0:
        raise RuntimeError(f"oracle_sconv_rollback: {STATUS.get(rc, rc)}")
    return out


# ----------------------------------------------------------------- FP8 KV cache ----

def e4m3_round(y: float) -> int:
    """Round a float64 to an OCP E4M3 code (nearest, ties to even, saturating at 448)."""
    return int(lib().oracle_e4m3_round(float(y)))


def e4m3_to_float(code: int) -> float:
    return float(lib().oracle_e4m3_to_double(int(code) & 0xFF))


def _u8(t) -> np.ndarray:
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint8
        return np.ascontiguousarray(t)
    assert t.dtype == torch.uint8 and t.device.type == "cpu"
    return t.contiguous().numpy()


def sconv_kv_fp8(k_raw, v_raw, w_k, w_v, state, cu_q_lens, slot_mapping, k_cache, v_cache,
                 k_scale: float, v_scale: float):
    """sconv_kv into FP8 caches (uint8 E4M3 codes, updated in place): code = e4m3(y / scale)."""
    for t in (k_cache, v_cache):
        assert t.is_contiguous() and t.dtype == torch.uint8 and t.device.type == "cpu"
    assert state.is_contiguous() and state.dtype == torch.bfloat16
    kr, vr = _u16(k_raw), _u16(v_raw)
    wk, wv = _arr(w_k, np.float32), _arr(w_v, np.float32)
    st = state.view(torch.int16).numpy().view(np.uint16)
    kc, vc = k_cache.numpy(), v_cache.numpy()
    cu = _arr(cu_q_lens, np.int32)
    sm = _arr(slot_mapping, np.int64)
    B = cu.shape[0] - 1
    T = kr.shape[0] if kr.ndim == 2 else 0
    rc = lib().oracle_sconv_kv_fp8(_ptr(kr), _ptr(vr), _ptr(wk), _ptr(wv), _ptr(st), _ptr(cu),
                                   _ptr(sm), _ptr(kc), _ptr(vc), float(k_scale), float(v_scale),
                                   B, T, kc.shape[1], kc.shape[0])
    if rc != 0:
        raise RuntimeError(f"oracle_sconv_kv_fp8: {STATUS.get(rc, rc)}")


def rel_attn_fp8(q, k_cache, v_cache, k_scale: float, v_scale: float, block_table, cu_q_lens,
                 seq_lens, bias, *, scale: float, window: int, rows=None, n_threads=None):
    """rel_attn over FP8 caches: K = e4m3(code) * k_scale, V = e4m3(code) * v_scale."""
    qa = _u16(q)
    kc, vc = _u8(k_cache), _u8(v_cache)
    bt = _arr(block_table, np.int32)
    cu = _arr(cu_q_lens, np.int32)
    sl = _arr(seq_lens, np.int32)
    bi = _arr(bias, np.float32)
    T, hq = qa.shape[0], qa.shape[1]
    rows = np.arange(T, dtype=np.int32) if rows is None else _arr(rows, np.int32)
    out = np.zeros((rows.shape[0], hq, 128), dtype=np.float64)
    lse = np.zeros((rows.shape[0], hq), dtype=np.float64)
    rc = lib().oracle_rel_attn_fp8(_ptr(qa), _ptr(kc), _ptr(vc), float(k_scale), float(v_scale),
                                   _ptr(bt), bt.shape[1], _ptr(cu), _ptr(sl), _ptr(bi),
                                   bi.shape[1], float(scale), int(window), cu.shape[0] - 1, T,
                                   hq, kc.shape[1], kc.shape[0], _ptr(rows), rows.shape[0],
                                   _ptr(out), _ptr(lse),
                                   host_cores() if n_threads is None else int(n_threads))
    if rc != 0:
        raise RuntimeError(f"oracle_rel_attn_fp8: {STATUS.get(rc, rc)}")
    return out, lse
