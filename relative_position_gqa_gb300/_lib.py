"""ctypes view of the C ABI in include/inkling.h (libinkling.so, built by build.py)."""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_build", "libinkling.so")

P = ctypes.c_void_p
I32 = ctypes.c_int32
I64 = ctypes.c_int64
F32 = ctypes.c_float
SZ = ctypes.c_size_t

# name -> argument types, in the order of include/inkling.h
SIGNATURES = {
    "inkling_sconv_kv": [P, P, P, P, P, P, P, P, P, I32, I32, I32, I64, I32, P, P],
    "inkling_sconv_kv_fp8": [P, P, P, P, P, P, P, P, P, F32, F32, I32, I32, I32, I64, I32, P, P],
    "inkling_sconv": [P, P, P, P, P, I32, I32, I32, I32, P, P],
    "inkling_sconv_state_rollback": [P, P, P, P, P, P, I32, I32, I32, I32, P, P],
    "inkling_rel_attn_prefill": [P, P, P, P, I32, P, P, P, I32, F32, I32, P, I32, P, I32, I32,
                                 I32, I32, I64, I32, P, P],
    "inkling_rel_attn_prefill_fp8_workspace_size": [I32, I32, I32, I32, I32, I32],
    "inkling_rel_attn_prefill_fp8": [P, P, P, F32, F32, P, I32, P, P, P, I32, F32, I32, P, I32,
                                     P, I32, I32, I32, I32, I64, I32, I32, P, SZ, P, P],
    "inkling_rel_attn_decode_workspace_size": [I32, I32, I32, I32, I32, I32, I32],
    "inkling_rel_attn_decode_plan": [I32, I32, I32, I32, I32, I32, I32, P],
    "inkling_rel_attn_decode": [P, P, P, P, I32, P, P, P, I32, F32, I32, P, I32, P, I32, I32,
                                I32, I32, I64, I32, I32, I32, P, SZ, P, P],
    "inkling_rel_attn_decode_sconv": [P, P, P, P, P, P, P, P, P, I32, P, P, P, I32, F32, I32, P,
                                      I32, P, I32, I32, I32, I32, I64, I32, I32, I32, P, SZ, P, P],
    "inkling_rel_attn_decode_fp8": [P, P, P, F32, F32, P, I32, P, P, P, I32, F32, I32, P, I32, P,
                                    I32, I32, I32, I32, I64, I32, I32, I32, P, SZ, P, P],
    "inkling_rel_attn_decode_noalloc_capacity": [],
    "inkling_rel_attn_decode_noalloc": [P, P, P, P, I32, P, P, P, I32, F32, I32, P, I32, P, I32,
                                        I32, I32, I32, I64, I32, I32, I32, P, P],
    "inkling_prefill_step_host": [P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, I32, P, P,
                                  I32, F32, I32, I32, P, I32, I32, I32, I32, I64, I32, I32, P,
                                  P, P, P, P],
    "inkling_decode_step_host": [P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, I32, P, P,
                                 I32, F32, I32, I32, P, I32, I32, I32, I32, I64, I32, I32, I32,
                                 P, SZ, I32, P, P, P, P],
    "inkling_prefill_step_host_fp8": [P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, F32, F32, P,
                                      I32, P, P, I32, F32, I32, I32, P, I32, I32, I32, I32, I64,
                                      I32, I32, P, SZ, I32, P, P, P, P, P],
    "inkling_decode_step_host_fp8": [P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, F32, F32, P,
                                     I32, P, P, I32, F32, I32, I32, P, I32, I32, I32, I32, I64,
                                     I32, I32, I32, P, SZ, I32, P, P, P, P],
    "inkling_selftest_bounded_wait": [I32, I32, P, P, P],
    "inkling_status_string": [ctypes.c_int],
    "inkling_version": [],
}
RESTYPES = {"inkling_rel_attn_decode_workspace_size": SZ,
            "inkling_rel_attn_prefill_fp8_workspace_size": SZ, "inkling_status_string": ctypes.c_char_p,
            "inkling_rel_attn_decode_noalloc_capacity": SZ}

_lib = None


class InklingError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn}: {status_string(code)} (status {code})")
        self.code = code


def library_path() -> str:
    return _SO


def load():
    """Load libinkling.so; raise if it has not been built (there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_SO):
            raise RuntimeError(
                f"Inkling CUDA library not built ({_SO} missing): run "
                "`python -m relative_position_gqa_gb300.build`")
        lib = ctypes.CDLL(_SO)
        for name, args in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = RESTYPES.get(name, ctypes.c_int)
        _lib = lib
    return _lib


def status_string(code: int) -> str:
    return load().inkling_status_string(int(code)).decode()


def _arg(x):
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return ctypes.c_void_p(x.data_ptr())
    return x


def call(name, *args):
    rc = getattr(load(), name)(*[_arg(a) for a in args])
    if rc != 0:
        raise InklingError(name, rc)


def workspace_size(*args) -> int:
    return int(load().inkling_rel_attn_decode_workspace_size(*[int(a) for a in args]))


def decode_plan(*args) -> list:
    plan = (ctypes.c_int32 * 4)()
    rc = load().inkling_rel_attn_decode_plan(*[int(a) for a in args], plan)
    if rc != 0:
        raise InklingError("inkling_rel_attn_decode_plan", rc)
    return list(plan)
