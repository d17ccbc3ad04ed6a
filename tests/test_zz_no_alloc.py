"""The allocation-free prefill entry point, kda_prefill_noalloc.

Some callers cannot allocate device memory: a serving host whose device
memory is already divided into its own pools, code that runs while a CUDA
graph is being captured, or a plugin that only receives tensors through the
C ABI.  kda_prefill_noalloc serves them with a scratch array built into the
library instead of a caller-provided workspace.  These tests check, through
the C ABI, that two calls in a row give the same results as kda_prefill with
its own workspace (within the parity tolerances used everywhere else), and
that a call too large for the built-in scratch is refused before anything
runs.  This file is collected last so that a run stopping at the first
failure has already run every other test; it also passes on its own in a
fresh process, where its first call is the one that looks up the scratch.
"""
import ctypes

import numpy as np
import pytest
import torch

from linear_attention_serving_gated_gb300 import build, inputs, kda
from tests.gpu_util import assert_o_close, assert_s_close, dev, dev_bf16, gates, host_f64

H = 16


def test_oversized_call_is_refused_without_launching():
    build.build()
    lib = kda.load()
    dummy = ctypes.c_void_p(0x10000)  # never dereferenced: the size check comes first
    gate = kda.kda_gate(None, None, -5.0, 1, 1, 128 ** -0.5)
    too_many = 4 * kda.PREFILL_STATIC_SCRATCH_BYTES // (16 * 131584) * 64
    st = lib.kda_prefill_noalloc(kda.dims(H), gate, dummy, dummy, dummy, dummy, dummy, too_many,
                                 dummy, 8, dummy, None, 1, too_many, dummy, None, None, None)
    assert st == kda.KDA_ERR_WORKSPACE


@pytest.mark.gpu
def test_noalloc_prefill_matches_workspace_prefill_on_two_calls():
    for seed, lens in ((70, [700, 1, 300]), (71, [1500])):
        T = sum(lens)
        d = inputs.prefill_inputs(seed=seed, lengths=lens, H=H, slots=8, gb_rows=T + 40)
        _, gg = gates(d, H=H)
        x = {n: dev_bf16(d[n]) for n in ("q", "k", "v", "g", "beta")}
        pool_ws = dev(d["pool"])
        pool_na = pool_ws.clone()
        idx, cu = dev(d["state_idx"]), dev(d["cu_seqlens"])
        o_ws = torch.empty((T, H, 128), dtype=torch.bfloat16, device="cuda")
        o_na = torch.full_like(o_ws, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        kda.kda_prefill(kda.dims(H), gg, x["q"], x["k"], x["v"], x["g"], x["beta"], pool_ws, idx,
                        cu, len(lens), o_ws)
        kda.kda_prefill_noalloc(kda.dims(H), gg, x["q"], x["k"], x["v"], x["g"], x["beta"], pool_na,
                                idx, cu, len(lens), o_na, err_flag=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        assert_o_close(o_na, host_f64(o_ws), "o (no-alloc vs workspace)")
        slots = [int(s) for s in d["state_idx"]]
        assert_s_close(pool_na[slots], host_f64(pool_ws[slots]), "final state (no-alloc vs workspace)")
        others = [s for s in range(8) if s not in slots]
        assert torch.equal(pool_na[others], pool_ws[others])
