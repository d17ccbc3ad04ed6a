"""Seeded synthetic inputs for the KDA serving path.

This module is the one piece shared by the CUDA path's tests/benchmark and the
CPU oracle's tests: it draws random numbers and encodes them, and holds none
of the method's arithmetic (no gate, norm or recurrence).

Distributions follow the pages' single-GPU microbenchmark setting ("[KDA]
Support Helion MTP verification and harden prefill, decode", sglang PR #42857,
Speed Tests and Profiling: 16 heads x 128, BF16 inputs, FP32 state, bounded
gate -5) with the concrete draws chosen for this library:

  q, k, v, gate input a, raw beta  ~ N(0, 1), rounded to BF16 (nearest-even),
                                   or to FP16 for the second precision
  A_log [HV] ~ U(-1, 1),  dt_bias [HV, K] ~ N(0, 0.1)   (FP32)
  state pool [slots, HV, V, K] ~ N(0, 0.02) in FP32 (or zero)
  varlen lengths U[1, 8192] with one length forced to 1, redrawn from the same
  stream until the total fits the padded bucket
  gate/beta padding rows: +-1e4 and NaN garbage (must never be read)

BF16 tensors are returned as int16 arrays of raw bit patterns, FP16 ones as
float16 arrays.
"""
from __future__ import annotations

import numpy as np

HEAD_DIM = 128


def bf16_bits(x) -> np.ndarray:
    """Round float32 values to BF16 (nearest-even) and return the bit patterns
    as int16.  NaN stays NaN."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        rounded[nan] = 0x7FC0
    return rounded.view(np.int16)


def encode16(x, dtype="bf16"):
    """float32 values -> the 16-bit token format: BF16 bit patterns (int16) or
    float16, both rounded to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return bf16_bits(x) if dtype == "bf16" else x.astype(np.float16)


def _normal16(rng, shape, dtype="bf16", std=1.0):
    x = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return encode16(x, dtype)


def _garbage16(rng, shape, dtype="bf16"):
    """Large-magnitude garbage for CUDA-graph bucket padding rows."""
    x = rng.choice(np.array([1e4, -1e4, np.nan, 3e4], dtype=np.float32), size=shape)
    return encode16(x, dtype)


def gate_params(rng, H, K=HEAD_DIM):
    A_log = rng.uniform(-1.0, 1.0, size=(H,)).astype(np.float32)
    dt_bias = (rng.standard_normal((H, K), dtype=np.float32) * np.float32(0.1)).astype(np.float32)
    return A_log, dt_bias


def state_pool(rng, slots, H, K=HEAD_DIM, V=HEAD_DIM, std=0.02, zero=False):
    if zero:
        return np.zeros((slots, H, V, K), dtype=np.float32)
    pool = rng.standard_normal((slots, H, V, K), dtype=np.float32)
    pool *= np.float32(std)
    return pool


def varlen_lengths(rng, n=8, max_len=8192, bucket=32768):
    """n lengths U[1, max_len], one forced to 1, redrawn until sum <= bucket."""
    while True:
        lens = rng.integers(1, max_len + 1, size=n)
        lens[rng.integers(0, n)] = 1
        if int(lens.sum()) <= bucket:
            return lens.astype(np.int64)


def prefill_inputs(seed=0, lengths=(128,), H=4, K=HEAD_DIM, V=HEAD_DIM, slots=4, gb_rows=None,
                   state_idx=None, zero_state=False, varlen=True, garbage=True, HV=None, dtype="bf16"):
    """Inputs of one prefill call.

    lengths: per-sequence token counts; varlen=False means the fixed layout
    (cu_seqlens absent, all lengths equal).  gb_rows >= sum(lengths) is the
    padded gate/beta row count.  HV (default H) value heads: q and k have H
    heads, everything else HV.  dtype: "bf16" (int16 bit patterns) or "f16"
    (float16) token tensors."""
    HV = H if HV is None else HV
    rng = np.random.default_rng(seed)
    lengths = np.asarray(lengths, dtype=np.int64)
    T = int(lengths.sum())
    gb_rows = T if gb_rows is None else int(gb_rows)
    assert gb_rows >= T
    A_log, dt_bias = gate_params(rng, HV, K)
    out = dict(
        q=_normal16(rng, (T, H, K), dtype),
        k=_normal16(rng, (T, H, K), dtype),
        v=_normal16(rng, (T, HV, V), dtype),
        g=np.empty((gb_rows, HV, K), dtype=np.int16 if dtype == "bf16" else np.float16),
        beta=np.empty((gb_rows, HV), dtype=np.int16 if dtype == "bf16" else np.float16),
        A_log=A_log, dt_bias=dt_bias,
    )
    out["g"][:T] = _normal16(rng, (T, HV, K), dtype)
    out["beta"][:T] = _normal16(rng, (T, HV), dtype)
    if gb_rows > T:
        if garbage:  # own stream, so the other inputs do not depend on it
            grng = np.random.default_rng([seed, 7919])
            out["g"][T:] = _garbage16(grng, (gb_rows - T, HV, K), dtype)
            out["beta"][T:] = _garbage16(grng, (gb_rows - T, HV), dtype)
        else:
            out["g"][T:] = 0
            out["beta"][T:] = 0
    out["pool"] = state_pool(rng, slots, HV, K, V, zero=zero_state)
    n = len(lengths)
    if state_idx is None:
        state_idx = rng.permutation(slots)[:n]
    out["state_idx"] = np.asarray(state_idx, dtype=np.int32)
    out["cu_seqlens"] = (np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
                         if varlen else None)
    out["lengths"] = lengths
    return out


def packed_rows(rng, rows, H, K=HEAD_DIM, V=HEAD_DIM, HV=None, dtype="bf16"):
    """rows of mixed_qkv [rows, 2*H*K + HV*V], gate input a [rows, HV*K], raw
    beta b [rows, HV], all in the 16-bit token format (HV defaults to H)."""
    HV = H if HV is None else HV
    return dict(
        mixed_qkv=_normal16(rng, (rows, 2 * H * K + HV * V), dtype),
        a=_normal16(rng, (rows, HV * K), dtype),
        b=_normal16(rng, (rows, HV), dtype),
    )


def decode_inputs(seed=0, B=16, H=16, K=HEAD_DIM, V=HEAD_DIM, slots=240, zero_state=False, HV=None,
                  dtype="bf16"):
    """One packed decode call: B requests gathered from a slots-deep pool by a
    random permutation prefix."""
    HV = H if HV is None else HV
    rng = np.random.default_rng(seed)
    A_log, dt_bias = gate_params(rng, HV, K)
    out = packed_rows(rng, B, H, K, V, HV, dtype)
    out.update(A_log=A_log, dt_bias=dt_bias,
               pool=state_pool(rng, slots, HV, K, V, zero=zero_state),
               state_idx=rng.permutation(slots)[:B].astype(np.int32))
    return out


def decode_step_rows(seed, step, B, H, K=HEAD_DIM, V=HEAD_DIM, HV=None, dtype="bf16"):
    """Fresh inputs for step `step` of a chained decode run."""
    return packed_rows(np.random.default_rng([seed, step]), B, H, K, V, HV, dtype)


def tree_parents(rng, B, T):
    """parent[0] = -1 and parent[i] ~ U{0..i-1}."""
    par = np.empty((B, T), dtype=np.int32)
    par[:, 0] = -1
    for i in range(1, T):
        par[:, i] = rng.integers(0, i, size=B)
    return par


def verify_inputs(seed=0, B=16, T=6, H=16, K=HEAD_DIM, V=HEAD_DIM, slots=240, zero_state=False,
                  HV=None, dtype="bf16"):
    """One verify call: B requests x T draft tokens, request-major rows."""
    HV = H if HV is None else HV
    rng = np.random.default_rng(seed)
    A_log, dt_bias = gate_params(rng, HV, K)
    out = packed_rows(rng, B * T, H, K, V, HV, dtype)
    out.update(A_log=A_log, dt_bias=dt_bias,
               pool=state_pool(rng, slots, HV, K, V, zero=zero_state),
               state_idx=rng.permutation(slots)[:B].astype(np.int32),
               parent=tree_parents(rng, B, T))
    return out
