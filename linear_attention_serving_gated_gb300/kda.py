"""ctypes binding of libkda (include/kda.h): the same entry points, taking
torch tensors on the GPU and marshalling them to device pointers.

Every step of the computation runs in the library's CUDA kernels; this
module only checks dtypes/devices, passes pointers, sizes and the current
stream, and raises ``KdaError`` on a non-OK status.  If ``libkda.so`` is
missing it raises at the first call: there is no other implementation.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkda.so")

KDA_OK = 0
KDA_ERR_NULL_ARG = 1
KDA_ERR_SHAPE = 2
KDA_ERR_UNSUPPORTED = 3
KDA_ERR_WORKSPACE = 4
KDA_ERR_CUDA = 5
KDA_ERR_ALIGNMENT = 6

KDA_DEVERR_SLOT = 1
KDA_DEVERR_PARENT = 2
KDA_DEVERR_SEQLENS = 4
KDA_DEVERR_ACCEPTED = 8
KDA_DEVERR_TIMEOUT = 16
KDA_DEVERR_INTERMEDIATE = 32

CHUNK = 64


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


KDA_DTYPE_BF16, KDA_DTYPE_F16 = 0, 1


class kda_dims(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("HV", ctypes.c_int), ("K", ctypes.c_int), ("V", ctypes.c_int),
                ("dtype", ctypes.c_int)]


class kda_gate(ctypes.Structure):
    _fields_ = [("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
                ("lower_bound", ctypes.c_float), ("beta_is_raw", ctypes.c_int),
                ("use_qk_l2norm", ctypes.c_int), ("scale", ctypes.c_float)]


EXPORTS = ("kda_status_string", "kda_prefill_workspace_size", "kda_prefill", "kda_decode_packed",
           "kda_verify_chain", "kda_verify_tree", "kda_commit", "kda_set_stage_events",
           "kda_prefill_noalloc", "kda_replay_ring_bytes", "kda_verify_chain_replay",
           "kda_commit_replay")

PREFILL_STATIC_SCRATCH_BYTES = 128 << 20  # KDA_PREFILL_STATIC_SCRATCH_BYTES in include/kda.h

_lib = None


def load(path: str = LIB_PATH):
    """Load libkda.so (built by build.py).  Raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"libkda.so not built ({path}); run linear_attention_serving_gated_gb300.build.build()")
        lib = ctypes.CDLL(path)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_status_string.argtypes = [i32]
        lib.kda_prefill_workspace_size.restype = sz
        lib.kda_prefill_workspace_size.argtypes = [kda_dims, i32, i64]
        lib.kda_prefill.restype = i32
        lib.kda_prefill.argtypes = [kda_dims, kda_gate, vp, vp, vp, vp, vp, i64, vp, i32, vp, vp, i32,
                                    i64, vp, vp, i64, vp, sz, vp, vp]
        lib.kda_decode_packed.restype = i32
        lib.kda_decode_packed.argtypes = [kda_dims, kda_gate, vp, i64, vp, vp, i32, vp, i32, vp, vp,
                                          vp, vp]
        lib.kda_verify_chain.restype = i32
        lib.kda_verify_chain.argtypes = [kda_dims, kda_gate, vp, i64, vp, vp, i32, i32, vp, i32, vp,
                                         vp, vp, vp, vp]
        lib.kda_verify_tree.restype = i32
        lib.kda_verify_tree.argtypes = [kda_dims, kda_gate, vp, i64, vp, vp, i32, i32, vp, vp, i32,
                                        vp, vp, vp, vp, vp]
        lib.kda_commit.restype = i32
        lib.kda_commit.argtypes = [kda_dims, vp, i32, i32, vp, vp, i32, vp, vp, vp]
        lib.kda_prefill_noalloc.restype = i32
        lib.kda_prefill_noalloc.argtypes = [kda_dims, kda_gate, vp, vp, vp, vp, vp, i64, vp, i32, vp,
                                            vp, i32, i64, vp, vp, i64, vp, vp]
        lib.kda_replay_ring_bytes.restype = sz
        lib.kda_replay_ring_bytes.argtypes = [kda_dims, i32, i32]
        lib.kda_verify_chain_replay.restype = i32
        lib.kda_verify_chain_replay.argtypes = [kda_dims, kda_gate, vp, i64, vp, vp, i32, i32, vp, i32,
                                                vp, vp, vp, vp, vp]
        lib.kda_commit_replay.restype = i32
        lib.kda_commit_replay.argtypes = [kda_dims, vp, i32, i32, vp, vp, i32, vp, vp, vp]
        lib.kda_set_stage_events.restype = None
        lib.kda_set_stage_events.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    try:
        return load().kda_status_string(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def _check(status: int, where: str):
    if status != KDA_OK:
        raise KdaError(status, where)


def _p(t):
    """Device pointer of a tensor (or None)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libkda takes device tensors")
    return ctypes.c_void_p(t.data_ptr())


def _in16(d, t, name):
    """A 16-bit token tensor: bfloat16 (or float16 when d.dtype is F16); int16
    raw bits are accepted either way."""
    want = torch.float16 if d.dtype == KDA_DTYPE_F16 else torch.bfloat16
    if t is not None and t.dtype not in (want, torch.int16):
        raise TypeError(f"{name} must be {want} (got {t.dtype})")
    return _p(t)


def _at_least(t, n, name, shape):
    """t must be dense (the library indexes it by its documented layout) and
    hold n elements (the rows the kernels touch); t None allowed."""
    if t is None:
        return
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() < n:
        raise ValueError(f"{name} must hold {shape} = {n} elements (got shape {tuple(t.shape)})")


def _packed_shapes(d, mixed_qkv, a, b, state_pool, state_idx, rows, reqs):
    """Shape rules of a packed-row call, checked on the host because the
    library sees only pointers.  As the pages' packed-decode validator does
    ("PR #35197 report: fix(kernel) Fix Helion small-token prefill bug",
    kda_decode.py snippet), HV, V and K come from the state's trailing
    dimensions and the gate input `a` must be [rows, HV*K]; every row the
    kernels read (rows = requests x tokens) must exist."""
    if state_pool.dim() < 3 or tuple(state_pool.shape[-3:]) != (d.HV, d.V, d.K):
        raise ValueError(f"state_pool must end in [HV, V, K] = [{d.HV}, {d.V}, {d.K}] "
                         f"(got {tuple(state_pool.shape)})")
    _at_least(state_pool, 0, "state_pool", "[slots, HV, V, K]")
    width = 2 * d.H * d.K + d.HV * d.V
    if mixed_qkv.dim() != 2 or mixed_qkv.shape[0] < rows or mixed_qkv.shape[1] < width \
            or mixed_qkv.stride(1) != 1:
        raise ValueError(f"mixed_qkv must be [>= {rows}, >= {width}] with unit column stride "
                         f"(got {tuple(mixed_qkv.shape)})")
    if a.shape[-1] != d.HV * d.K or a.numel() < rows * d.HV * d.K or not a.is_contiguous():
        raise ValueError(f"`a` must have shape [B, HV*K] = [{rows}, {d.HV * d.K}], contiguous "
                         f"(got {tuple(a.shape)})")
    if b.numel() < rows * d.HV or not b.is_contiguous():
        raise ValueError(f"`b` must have shape [B, HV] = [{rows}, {d.HV}], contiguous "
                         f"(got {tuple(b.shape)})")
    _at_least(state_idx, reqs, "state_idx", f"[{reqs}]")


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


class Gate:
    """Fold options of a call (kda_gate): A_log [HV] / dt_bias [HV*K] FP32
    device tensors or None, lower_bound (None = unbounded, rejected when
    A_log is given), beta_is_raw, use_qk_l2norm, scale."""

    def __init__(self, A_log=None, dt_bias=None, lower_bound=-5.0, beta_is_raw=True,
                 use_qk_l2norm=True, scale=128 ** -0.5):
        self.A_log, self.dt_bias = A_log, dt_bias
        self.lower_bound = lower_bound
        self.beta_is_raw, self.use_qk_l2norm, self.scale = beta_is_raw, use_qk_l2norm, scale

    def c(self):
        for t in (self.A_log, self.dt_bias):
            if t is not None and t.dtype != torch.float32:
                raise TypeError("A_log and dt_bias must be float32")
        lb = float("nan") if self.lower_bound is None else float(self.lower_bound)
        return kda_gate(_p(self.A_log), _p(self.dt_bias), lb, int(bool(self.beta_is_raw)),
                        int(bool(self.use_qk_l2norm)), float(self.scale))


def dims(H, K=128, V=128, HV=None, dtype=KDA_DTYPE_BF16):
    """Head counts and sizes of a call; dtype: element type of the 16-bit
    token tensors and of o (KDA_DTYPE_BF16 or KDA_DTYPE_F16)."""
    return kda_dims(int(H), int(HV if HV is not None else H), int(K), int(V), int(dtype))


def kda_prefill_workspace_size(d: kda_dims, num_seqs: int, total_tokens: int) -> int:
    return int(load().kda_prefill_workspace_size(d, int(num_seqs), int(total_tokens)))


def _intermediate_chunks(d, intermediate):
    """Chunk records an intermediate-state buffer holds: it must be a dense
    [chunks, HV, V, K] FP32 tensor.  The library writes only that many (the
    chunk count follows cu_seqlens, which is on the device) and flags the
    rest."""
    if intermediate is None:
        return 0
    if intermediate.dtype != torch.float32 or intermediate.dim() != 4 or \
            tuple(intermediate.shape[1:]) != (d.HV, d.V, d.K):
        raise ValueError(f"intermediate must be float32 [chunks, HV, V, K] = [*, {d.HV}, {d.V}, {d.K}] "
                         f"(got {intermediate.dtype} {tuple(intermediate.shape)})")
    _at_least(intermediate, 0, "intermediate", "[chunks, HV, V, K]")
    return int(intermediate.shape[0])


def _prefill_shapes(d, q, k, v, g, beta, state_pool, state_idx, cu_seqlens, num_seqs, o):
    """Every element the prefill kernels touch for T = q.shape[0] tokens and
    gb_rows = g.shape[0] gate rows must exist (the library sees pointers)."""
    T, gb_rows, n = q.shape[0], g.shape[0], int(num_seqs)
    if state_pool.dim() < 3 or tuple(state_pool.shape[-3:]) != (d.HV, d.V, d.K):
        raise ValueError(f"state_pool must end in [HV, V, K] = [{d.HV}, {d.V}, {d.K}] "
                         f"(got {tuple(state_pool.shape)})")
    _at_least(state_pool, 0, "state_pool", "[slots, HV, V, K]")
    _at_least(q, T * d.H * d.K, "q", f"[{T}, H, K]")
    _at_least(k, T * d.H * d.K, "k", f"[{T}, H, K]")
    _at_least(v, T * d.HV * d.V, "v", f"[{T}, HV, V]")
    _at_least(g, gb_rows * d.HV * d.K, "g", f"[{gb_rows}, HV, K]")
    _at_least(beta, gb_rows * d.HV, "beta", f"[{gb_rows}, HV]")
    _at_least(o, T * d.HV * d.V, "o", f"[{T}, HV, V]")
    _at_least(state_idx, n, "state_idx", f"[{n}]")
    _at_least(cu_seqlens, n + 1, "cu_seqlens", f"[{n + 1}]")


def kda_prefill(d, gate: Gate, q, k, v, g, beta, state_pool, state_idx, cu_seqlens, num_seqs,
                o, intermediate=None, workspace=None, err_flag=None, stream=None):
    """Chunked varlen prefill (see kda.h).  q,k [T,H,K], v [T,HV,V], g
    [gb_rows,HV,K], beta [gb_rows,HV] bf16; state_pool [slots,HV,V,K] fp32
    (in place); o [T,HV,V] bf16 (written)."""
    T = q.shape[0]
    gb_rows = g.shape[0]
    _prefill_shapes(d, q, k, v, g, beta, state_pool, state_idx, cu_seqlens, num_seqs, o)
    inter_chunks = _intermediate_chunks(d, intermediate)
    if workspace is None:
        need = kda_prefill_workspace_size(d, num_seqs, T)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = load().kda_prefill(
        d, gate.c(), _in16(d, q, "q"), _in16(d, k, "k"), _in16(d, v, "v"), _in16(d, g, "g"), _in16(d, beta, "beta"),
        int(gb_rows), _p(state_pool), int(state_pool.shape[0]), _p(state_idx), _p(cu_seqlens),
        int(num_seqs), int(T), _in16(d, o, "o"), _p(intermediate), inter_chunks, _p(workspace),
        int(workspace.numel() * workspace.element_size()), _p(err_flag), _stream(stream))
    _check(st, "kda_prefill")


def kda_prefill_noalloc(d, gate: Gate, q, k, v, g, beta, state_pool, state_idx, cu_seqlens,
                        num_seqs, o, intermediate=None, err_flag=None, stream=None):
    """kda_prefill with the library's built-in static scratch (see kda.h): for
    callers that cannot allocate device memory."""
    _prefill_shapes(d, q, k, v, g, beta, state_pool, state_idx, cu_seqlens, num_seqs, o)
    inter_chunks = _intermediate_chunks(d, intermediate)
    st = load().kda_prefill_noalloc(
        d, gate.c(), _in16(d, q, "q"), _in16(d, k, "k"), _in16(d, v, "v"), _in16(d, g, "g"), _in16(d, beta, "beta"),
        int(g.shape[0]), _p(state_pool), int(state_pool.shape[0]), _p(state_idx), _p(cu_seqlens),
        int(num_seqs), int(q.shape[0]), _in16(d, o, "o"), _p(intermediate), inter_chunks,
        _p(err_flag), _stream(stream))
    _check(st, "kda_prefill_noalloc")


def kda_decode_packed(d, gate: Gate, mixed_qkv, a, b, state_pool, state_idx, o, err_flag=None,
                      stream=None):
    B = mixed_qkv.shape[0]
    _packed_shapes(d, mixed_qkv, a, b, state_pool, state_idx, B, B)
    _at_least(o, B * d.HV * d.V, "o", f"[{B}, HV, V]")
    st = load().kda_decode_packed(
        d, gate.c(), _in16(d, mixed_qkv, "mixed_qkv"), int(mixed_qkv.stride(0)), _in16(d, a, "a"),
        _in16(d, b, "b"), int(mixed_qkv.shape[0]), _p(state_pool), int(state_pool.shape[0]),
        _p(state_idx), _in16(d, o, "o"), _p(err_flag), _stream(stream))
    _check(st, "kda_decode_packed")


def _verify_shapes(d, mixed_qkv, a, b, B, T, state_pool, state_idx, o):
    rows = int(B) * int(T)
    _packed_shapes(d, mixed_qkv, a, b, state_pool, state_idx, rows, int(B))
    _at_least(o, rows * d.HV * d.V, "o", f"[{B}, {T}, HV, V]")


def kda_verify_chain(d, gate: Gate, mixed_qkv, a, b, B, T, state_pool, state_idx, o, snapshots,
                     err_flag=None, stream=None):
    _verify_shapes(d, mixed_qkv, a, b, B, T, state_pool, state_idx, o)
    _at_least(snapshots, B * T * d.HV * d.V * d.K, "snapshots", f"[{B}, {T}, HV, V, K]")
    st = load().kda_verify_chain(
        d, gate.c(), _in16(d, mixed_qkv, "mixed_qkv"), int(mixed_qkv.stride(0)), _in16(d, a, "a"),
        _in16(d, b, "b"), int(B), int(T), _p(state_pool), int(state_pool.shape[0]), _p(state_idx),
        _in16(d, o, "o"), _p(snapshots), _p(err_flag), _stream(stream))
    _check(st, "kda_verify_chain")


def kda_verify_tree(d, gate: Gate, mixed_qkv, a, b, B, T, parent_idx, state_pool, state_idx, o,
                    snapshots, err_flag=None, stream=None):
    _verify_shapes(d, mixed_qkv, a, b, B, T, state_pool, state_idx, o)
    _at_least(snapshots, B * T * d.HV * d.V * d.K, "snapshots", f"[{B}, {T}, HV, V, K]")
    _at_least(parent_idx, B * T, "parent_idx", f"[{B}, {T}]")
    st = load().kda_verify_tree(
        d, gate.c(), _in16(d, mixed_qkv, "mixed_qkv"), int(mixed_qkv.stride(0)), _in16(d, a, "a"),
        _in16(d, b, "b"), int(B), int(T), _p(parent_idx), _p(state_pool), int(state_pool.shape[0]),
        _p(state_idx), _in16(d, o, "o"), _p(snapshots), _p(err_flag), _stream(stream))
    _check(st, "kda_verify_tree")


def kda_commit(d, snapshots, B, T, accepted, state_pool, state_idx, err_flag=None, stream=None):
    _at_least(snapshots, B * T * d.HV * d.V * d.K, "snapshots", f"[{B}, {T}, HV, V, K]")
    _at_least(accepted, B, "accepted", f"[{B}]")
    _at_least(state_idx, B, "state_idx", f"[{B}]")
    st = load().kda_commit(d, _p(snapshots), int(B), int(T), _p(accepted), _p(state_pool),
                           int(state_pool.shape[0]), _p(state_idx), _p(err_flag), _stream(stream))
    _check(st, "kda_commit")


def kda_replay_ring_bytes(d, B, T) -> int:
    return int(load().kda_replay_ring_bytes(d, int(B), int(T)))


def kda_verify_chain_replay(d, gate: Gate, mixed_qkv, a, b, B, T, state_pool, state_idx, o, ring,
                            err_flag=None, stream=None):
    """Chain verify without snapshots: o as kda_verify_chain, each token's
    folded inputs recorded in `ring` (kda_replay_ring_bytes bytes, FP32)."""
    _verify_shapes(d, mixed_qkv, a, b, B, T, state_pool, state_idx, o)
    _at_least(ring, kda_replay_ring_bytes(d, B, T) // 4, "ring", "kda_replay_ring_bytes / 4 FP32")
    st = load().kda_verify_chain_replay(
        d, gate.c(), _in16(d, mixed_qkv, "mixed_qkv"), int(mixed_qkv.stride(0)), _in16(d, a, "a"),
        _in16(d, b, "b"), int(B), int(T), _p(state_pool), int(state_pool.shape[0]), _p(state_idx),
        _in16(d, o, "o"), _p(ring), _p(err_flag), _stream(stream))
    _check(st, "kda_verify_chain_replay")


def kda_commit_replay(d, ring, B, T, accepted, state_pool, state_idx, err_flag=None, stream=None):
    """Advances each request's pool state through its accepted draft tokens
    from the ring written by kda_verify_chain_replay."""
    _at_least(ring, kda_replay_ring_bytes(d, B, T) // 4, "ring", "kda_replay_ring_bytes / 4 FP32")
    _at_least(accepted, B, "accepted", f"[{B}]")
    _at_least(state_idx, B, "state_idx", f"[{B}]")
    st = load().kda_commit_replay(d, _p(ring), int(B), int(T), _p(accepted), _p(state_pool),
                                  int(state_pool.shape[0]), _p(state_idx), _p(err_flag),
                                  _stream(stream))
    _check(st, "kda_commit_replay")


def kda_set_stage_events(events=None):
    """Profiling aid: torch.cuda.Event triple recorded by every later call
    (before its first kernel, between the prefill's two kernels, after its
    last kernel); a None entry is not recorded; None clears all three."""
    if events is None:
        load().kda_set_stage_events(None)
        return
    arr = (ctypes.c_void_p * 3)(*[ctypes.c_void_p(e.cuda_event if e is not None else None)
                                  for e in events])
    load().kda_set_stage_events(arr)
