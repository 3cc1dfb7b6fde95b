"""ctypes declarations of the C ABI in include/engram.h and include/engram_synth.h.

Loading fails loudly when the in-tree libraries have not been built: there is no
fallback path.  Build them with ``python -m engram_hashed_gram_gb300.build``
(or ``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int32, c_int64, c_uint64, c_void_p

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

ENGRAM_OK = 0
ENGRAM_EINVAL = -1
ENGRAM_ENOMEM = -2
ENGRAM_ECUDA = -3
ENGRAM_ERANGE = -4
ENGRAM_ETIMEOUT = -5
ENGRAM_EUNSUPPORTED = -6

NOALLOC_MAX_TOKENS = 64          # ENGRAM_NOALLOC_MAX_TOKENS
NOALLOC_SCRATCH_BYTES = 20529408  # ENGRAM_NOALLOC_SCRATCH_BYTES

SCALE_F32 = 0
SCALE_E8M0 = 1
WKV_BF16 = 0
WKV_MXFP8 = 1
TEST_HOLD_GATE_FLAGS = 1


class EngramConfig(ctypes.Structure):
    _fields_ = [
        ("dim", c_int32),
        ("hc_mult", c_int32),
        ("n_cols", c_int32),
        ("head_dim", c_int32),
        ("scale_block", c_int32),
        ("scale_fmt", c_int32),
        ("num_rows", c_int64),
        ("eps", c_float),
        ("clamp", c_float),
        ("max_tokens", c_int32),
        ("check_ids", c_int32),
        ("fuse_gate", c_int32),
        ("wkv_fmt", c_int32),
        ("row_offset", c_int64),
    ]


class EngramPlanInfo(ctypes.Structure):
    _fields_ = [
        ("splits", c_int32),
        ("ctas", c_int32),
        ("cta_pairs", c_int32),
        ("rem_tiles", c_int32),
        ("rem_splits", c_int32),
        ("fused_gate", c_int32),
    ]


class EngramHashConfig(ctypes.Structure):
    _fields_ = [
        ("n_layers", c_int32),
        ("max_ngram_size", c_int32),
        ("n_heads", c_int32),
        ("max_batch", c_int32),
        ("max_len", c_int64),
        ("vocab_size", c_int64),
        ("pad_id", c_int32),
        ("dead_id", c_int32),
    ]


class EngramWeights(ctypes.Structure):
    _fields_ = [
        ("table", c_void_p),
        ("scale", c_void_p),
        ("wkv", c_void_p),
        ("q_weight", c_void_p),
        ("k_weight", c_void_p),
        ("wkv_scale", c_void_p),
    ]


# name -> (restype, argtypes); every function declared in include/engram.h
ENGRAM_FUNCS = {
    "engram_create": (c_int32, [POINTER(c_void_p), POINTER(EngramConfig), POINTER(EngramWeights)]),
    "engram_destroy": (None, [c_void_p]),
    "engram_forward": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_void_p]),
    "engram_lookup_project": (c_int32, [c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_void_p]),
    "engram_gate_apply": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int64,
                                    c_void_p]),
    "engram_lookup": (c_int32, [c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_void_p]),
    "engram_forward_rows": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_void_p]),
    "engram_sync_status": (c_int32, [c_void_p, c_void_p, POINTER(c_int64)]),
    "engram_plan": (c_int32, [c_void_p, c_int64, POINTER(c_int32), POINTER(c_int32)]),
    "engram_forward_kernels": (c_int32, [c_void_p, c_int64, POINTER(c_int32)]),
    "engram_describe_plan": (c_int32, [c_void_p, c_int64, POINTER(EngramPlanInfo)]),
    "engram_set_sm_budget": (c_int32, [c_void_p, c_int32]),
    "engram_test_hook": (c_int32, [c_void_p, c_int32]),
    "engram_forward_noalloc": (c_int32, [POINTER(EngramConfig), POINTER(EngramWeights), c_void_p, c_void_p,
                                         c_void_p, c_void_p, c_int64, c_int64, c_void_p]),
    "engram_hash": (c_int32, [POINTER(EngramHashConfig), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                              c_void_p, c_int64, c_void_p, c_int64, c_int64, c_void_p]),
    "engram_enable_stage_timing": (c_int32, [c_void_p, c_int32]),
    "engram_stage_times": (c_int32, [c_void_p, POINTER(c_float)]),
    "engram_stage_times_n": (c_int32, [c_void_p, c_int32, POINTER(c_float)]),
    "engram_status_string": (c_char_p, [c_int32]),
    "engram_abi_version": (c_int32, []),
}

SYNTH_FUNCS = {
    "engram_synth_fill_table": (c_int32, [c_void_p, c_void_p, c_int64, c_int64, c_int32, c_int32, c_uint64, c_uint64,
                                          c_void_p, c_void_p, c_void_p]),
    "engram_synth_fill_scales_e8m0": (c_int32, [c_void_p, c_int64, c_int64, c_int32, c_int32, c_uint64, c_void_p,
                                                c_void_p]),
}

_LIBS: dict[str, ctypes.CDLL] = {}


def lib_file(name: str) -> str:
    return os.path.join(HERE, name)


def _load(name: str, funcs: dict) -> ctypes.CDLL:
    if name in _LIBS:
        return _LIBS[name]
    path = lib_file(name)
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: the Engram CUDA library has not been built "
            "(run `python -m engram_hashed_gram_gb300.build`); there is no fallback path")
    lib = ctypes.CDLL(path)
    for fname, (res, args) in funcs.items():
        f = getattr(lib, fname)
        f.restype = res
        f.argtypes = args
    _LIBS[name] = lib
    return lib


def engram() -> ctypes.CDLL:
    return _load("libengram.so", ENGRAM_FUNCS)


def synth() -> ctypes.CDLL:
    return _load("libengram_synth.so", SYNTH_FUNCS)


class EngramError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = engram().engram_status_string(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")


def check(status: int, where: str) -> None:
    if status != ENGRAM_OK:
        raise EngramError(status, where)
