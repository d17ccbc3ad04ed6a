"""Python access to the FP64 CPU oracle of the KDA gated delta-rule path.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU-baseline leg
of the benchmark load this module; the library itself never does.  It shares
no code with the CUDA path.

All arithmetic lives in ``kda_oracle.c`` (built here into
``libkda_oracle.so``).  This module only marshals numpy arrays: BF16 inputs
arrive as raw 16-bit patterns and are widened exactly to float32; states are
float64 throughout; outputs come back as float64.

The contracts follow the pages:
  * prefill -- ``chunk_kda`` of the report "PR #35197: fix(kernel) Fix Helion
    small-token prefill bug" (key source snippet of kda_prefill.py): an indexed
    pool is required and gate/beta rows past the token count are padding.
  * decode -- ``validate_packed_decode_inputs`` in the same report: packed
    ``mixed_qkv`` rows and gate input ``a`` of width HV*K.
  * verify/commit -- "[KDA] Support Helion MTP verification and harden
    prefill, decode" (sglang PR #42857), Modifications and the two-round
    verify/commit review thread.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB = os.path.join(_HERE, "libkda_oracle.so")

CHUNK = 64


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-Wall", "-Werror", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
             "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


class _Params(ctypes.Structure):
    _fields_ = [
        ("H", ctypes.c_int), ("HV", ctypes.c_int), ("K", ctypes.c_int), ("V", ctypes.c_int),
        ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("lower_bound", ctypes.c_double), ("beta_is_raw", ctypes.c_int),
        ("use_qk_l2norm", ctypes.c_int), ("scale", ctypes.c_double),
    ]


_lib = None


def _load():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        for name in ("kdao_prefill", "kdao_decode", "kdao_verify", "kdao_commit"):
            getattr(_lib, name).restype = ctypes.c_int
    return _lib


class OracleError(RuntimeError):
    pass


_ERRORS = {1: "bad argument", 2: "bad or duplicate state slot", 3: "bad tree parent",
           4: "bad cu_seqlens", 5: "out of memory"}


def _check(rc: int):
    if rc:
        raise OracleError(_ERRORS.get(rc, "error %d" % rc))


def bf16_to_f32(x) -> np.ndarray:
    """Widen raw BF16 bit patterns (int16/uint16 array) to float32, exactly."""
    x = np.asarray(x)
    if x.dtype in (np.int16, np.uint16):
        return (x.astype(np.uint16).astype(np.uint32) << 16).view(np.float32)
    return np.ascontiguousarray(x, dtype=np.float32)


def _f32(x):
    return None if x is None else np.ascontiguousarray(bf16_to_f32(x), dtype=np.float32)


def _i32(x):
    return None if x is None else np.ascontiguousarray(np.asarray(x), dtype=np.int32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Gate:
    """Fold parameters of one call: the gate, beta and q/k normalisation."""

    def __init__(self, H, K, V, HV=None, A_log=None, dt_bias=None, lower_bound=-5.0,
                 beta_is_raw=True, use_qk_l2norm=True, scale=None):
        self.H, self.K, self.V = int(H), int(K), int(V)
        self.HV = int(HV if HV is not None else H)
        self.A_log = None if A_log is None else np.ascontiguousarray(A_log, dtype=np.float32)
        self.dt_bias = None if dt_bias is None else np.ascontiguousarray(dt_bias, dtype=np.float32)
        self.lower_bound = float(lower_bound)
        self.beta_is_raw = bool(beta_is_raw)
        self.use_qk_l2norm = bool(use_qk_l2norm)
        self.scale = float(scale if scale is not None else self.K ** -0.5)

    def _c(self):
        return _Params(self.H, self.HV, self.K, self.V, _ptr(self.A_log), _ptr(self.dt_bias),
                       self.lower_bound, int(self.beta_is_raw), int(self.use_qk_l2norm),
                       self.scale)


def _threads(n):
    return int(n) if n else (os.cpu_count() or 1)


def prefill(gate: Gate, q, k, v, g, beta, pool, state_idx, cu_seqlens=None, num_seqs=None,
            intermediate=False, chunk=CHUNK, nthreads=None):
    """Token-by-token prefill.  ``pool`` (float64 [slots,HV,V,K]) is updated in
    place.  Returns ``o`` [T,HV,V] and, if asked, the chunk-start states."""
    q, k, v, g, beta = (_f32(x) for x in (q, k, v, g, beta))
    T = q.shape[0]
    gb_rows = g.shape[0]
    assert pool.dtype == np.float64 and pool.flags.c_contiguous
    state_idx = _i32(state_idx)
    cu = _i32(cu_seqlens)
    n = int(num_seqs if num_seqs is not None else (len(cu) - 1 if cu is not None else len(state_idx)))
    if cu is not None:
        lens = np.diff(cu)
    else:
        lens = np.full(n, T // n)
    nchunks = int(sum((int(x) + chunk - 1) // chunk for x in lens))
    o = np.zeros((T, gate.HV, gate.V), dtype=np.float64)
    inter = np.zeros((nchunks, gate.HV, gate.V, gate.K), dtype=np.float64) if intermediate else None
    p = gate._c()
    _check(_load().kdao_prefill(
        ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), ctypes.c_long(gb_rows),
        _ptr(pool), ctypes.c_int(pool.shape[0]), _ptr(state_idx), _ptr(cu), ctypes.c_int(n),
        ctypes.c_long(T), ctypes.c_int(chunk), _ptr(o), _ptr(inter),
        ctypes.c_int(_threads(nthreads))))
    return (o, inter) if intermediate else o


def decode(gate: Gate, mixed_qkv, a, b, pool, state_idx, nthreads=None):
    """One packed decode step per request; ``pool`` updated in place."""
    x, a, b = _f32(mixed_qkv), _f32(a), _f32(b)
    B = x.shape[0]
    state_idx = _i32(state_idx)
    o = np.zeros((B, gate.HV, gate.V), dtype=np.float64)
    p = gate._c()
    _check(_load().kdao_decode(
        ctypes.byref(p), _ptr(x), ctypes.c_long(x.shape[1]), _ptr(a), _ptr(b), ctypes.c_int(B),
        _ptr(pool), ctypes.c_int(pool.shape[0]), _ptr(state_idx), _ptr(o),
        ctypes.c_int(_threads(nthreads))))
    return o


def verify(gate: Gate, mixed_qkv, a, b, B, T, pool, state_idx, parent=None, nthreads=None):
    """Chain (parent None) or tree verify.  The pool is read only.
    Returns ``o`` [B,T,HV,V] and ``snapshots`` [B,T,HV,V,K]."""
    x, a, b = _f32(mixed_qkv), _f32(a), _f32(b)
    state_idx = _i32(state_idx)
    par = _i32(parent)
    o = np.zeros((B, T, gate.HV, gate.V), dtype=np.float64)
    snaps = np.zeros((B, T, gate.HV, gate.V, gate.K), dtype=np.float64)
    p = gate._c()
    _check(_load().kdao_verify(
        ctypes.byref(p), _ptr(x), ctypes.c_long(x.shape[1]), _ptr(a), _ptr(b), ctypes.c_int(B),
        ctypes.c_int(T), _ptr(par), _ptr(pool), ctypes.c_int(pool.shape[0]), _ptr(state_idx),
        _ptr(o), _ptr(snaps), ctypes.c_int(_threads(nthreads))))
    return o, snaps


def commit(snapshots, accepted, pool, state_idx):
    """pool[state_idx[b]] <- snapshots[b, accepted[b]] where accepted[b] >= 0."""
    snapshots = np.ascontiguousarray(snapshots, dtype=np.float64)
    B, T, HV, V, K = snapshots.shape
    acc, idx = _i32(accepted), _i32(state_idx)
    _check(_load().kdao_commit(_ptr(snapshots), ctypes.c_int(B), ctypes.c_int(T), ctypes.c_int(HV),
                               ctypes.c_int(V), ctypes.c_int(K), _ptr(acc), _ptr(pool),
                               ctypes.c_int(pool.shape[0]), _ptr(idx)))
