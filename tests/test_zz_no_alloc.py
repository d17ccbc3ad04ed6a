"""The allocation-free prefill entry point, kda_prefill_noalloc.

Some callers cannot allocate device memory: a serving host whose device
memory is already divided into its own pools, code that runs while a CUDA
graph is being captured, or a plugin that only receives tensors through the
C ABI.  kda_prefill_noalloc serves them with a scratch array built into the
library instead of a caller-provided workspace.  These tests check, through
the C ABI, that two calls in a row give the same bits as kda_prefill with its
own workspace (both run the same kernels on the same inputs), and that a call
too large for the built-in scratch is refused before anything runs, at
exactly the size kda.h states.  This file is collected last so that a run
stopping at the first failure has already run every other test; it also
passes on its own in a fresh process, where its first call is the one that
looks up the scratch.
"""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

from linear_attention_serving_gated_gb300 import build, inputs, kda
from tests.gpu_util import dev, dev_bf16, gates

H = 16
HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "kda.h")
DUMMY = ctypes.c_void_p(0x10000)  # never dereferenced: every call below returns before a launch


def _lib():
    build.build()
    return kda.load()


def test_scratch_size_constant_matches_the_header():
    text = open(HEADER).read()
    m = re.search(r"#define\s+KDA_PREFILL_STATIC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", text)
    assert m, "KDA_PREFILL_STATIC_SCRATCH_BYTES not found in kda.h"
    assert int(m.group(1)) << int(m.group(2)) == kda.PREFILL_STATIC_SCRATCH_BYTES


def _noalloc_status(lib, T, pool):
    """Status of a one-sequence, 16-head call of T tokens.  With pool = NULL
    a call that passes the scratch-size check stops at the pool check (or, on
    a machine without a GPU, at the device lookup), before any launch."""
    gate = kda.kda_gate(None, None, -5.0, 1, 1, 128 ** -0.5)
    return lib.kda_prefill_noalloc(kda.dims(H), gate, DUMMY, DUMMY, DUMMY, DUMMY, DUMMY, T, pool, 8,
                                   DUMMY, None, 1, T, DUMMY, None, 0, None, None)


def _largest_fitting_tokens(lib):
    """Largest one-sequence token count whose workspace fits the scratch,
    from the library's own size function."""
    d = kda.dims(H)
    lo, hi = 0, 1 << 20
    assert lib.kda_prefill_workspace_size(d, 1, hi) > kda.PREFILL_STATIC_SCRATCH_BYTES
    while lo + 1 < hi:
        mid = (lo + hi) // 2
        if lib.kda_prefill_workspace_size(d, 1, mid) <= kda.PREFILL_STATIC_SCRATCH_BYTES:
            lo = mid
        else:
            hi = mid
    return lo


def test_size_limit_is_the_documented_rule():
    lib = _lib()
    t_max = _largest_fitting_tokens(lib)
    assert t_max == 2943  # 46 records per head at 16 heads, as kda.h states
    assert _noalloc_status(lib, t_max, None) != kda.KDA_ERR_WORKSPACE
    assert _noalloc_status(lib, t_max + 1, None) == kda.KDA_ERR_WORKSPACE
    # the pages' 1 x 4096 shape at 16 heads does not fit
    assert _noalloc_status(lib, 4096, DUMMY) == kda.KDA_ERR_WORKSPACE


@pytest.mark.gpu
def test_noalloc_prefill_matches_workspace_prefill_on_two_calls():
    for seed, lens, given_decay in ((70, [700, 1, 300], False), (71, [1500], True)):
        T = sum(lens)
        d = inputs.prefill_inputs(seed=seed, lengths=lens, H=H, slots=8, gb_rows=T + 40)
        if given_decay:  # the path that uses the scratch's per-sequence flags
            d["g"][:T] = inputs.encode16(-0.5 * np.random.default_rng(seed).random((T, H, 128)))
            d["A_log"] = None
        _, gg = gates(d, H=H) if d["A_log"] is not None else (None, kda.Gate())
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
        assert torch.equal(o_na, o_ws), "o differs between the no-alloc and workspace calls"
        assert torch.equal(pool_na, pool_ws), "pool differs between the no-alloc and workspace calls"
