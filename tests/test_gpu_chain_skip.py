"""GPU parity of the state pass's skipped chain products, through the C ABI,
against the FP64 oracle.

A chunk's end state is S_end = M_c S + B_c ("[KDA] Support Helion MTP
verification and harden prefill, decode", the chunked form of the gated
delta rule).  The pass leaves the product M_c S out only where it cannot
change an FP32 bit of S_end: M_c all zero (the transform then stores no M_c),
or 128 max|M_c| max|S| below a quarter of half an ulp of every element of
B_c.  These tests mix the three cases inside one sequence and check that a
tiny map is still applied when the state is large enough for it to matter.
"""
import numpy as np
import pytest
import torch

from linear_attention_serving_gated_gb300 import inputs, kda
from oracle import kda_oracle as ko
from tests.gpu_util import assert_o_close, assert_s_close, dev, dev_bf16, gates

pytestmark = pytest.mark.gpu

K = 128


def _run(d, H, og, gg):
    lens = d["lengths"]
    T = int(lens.sum())
    x = {n: dev_bf16(d[n]) for n in ("q", "k", "v", "g", "beta")}
    pool = dev(d["pool"])
    o = torch.full((T, H, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    nch = int(sum((int(L) + 63) // 64 for L in lens))
    inter = torch.full((nch, H, K, K), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_prefill(kda.dims(H), gg, x["q"], x["k"], x["v"], x["g"], x["beta"], pool, dev(d["state_idx"]),
                    dev(d["cu_seqlens"]), len(lens), o, inter, err_flag=err)
    torch.cuda.synchronize()
    opool = d["pool"].astype(np.float64)
    o_ref, inter_ref = ko.prefill(og, d["q"], d["k"], d["v"], d["g"], d["beta"], opool, d["state_idx"],
                                  d["cu_seqlens"], intermediate=True)
    assert int(err.item()) == 0, f"device error bits {int(err.item())}"
    slots = [int(s) for s in d["state_idx"] if s >= 0]
    return o, o_ref, pool[slots], opool[slots], inter, inter_ref


def test_zero_tiny_and_full_maps_in_one_sequence():
    """Given log-decays chosen per chunk: about -5 per token (the map
    underflows to zero in FP32), about -1 per token (a tiny nonzero map, left
    out next to an O(1) state) and about -0.01 per token (the map keeps the
    state, so the product runs), in a repeating pattern over 21 chunks plus a
    ragged tail, next to a second, shorter sequence."""
    H, lens = 4, [21 * 64 + 37, 300]
    T = sum(lens)
    d = inputs.prefill_inputs(seed=330, lengths=lens, H=H, slots=6, gb_rows=T + 16)
    rng = np.random.default_rng(331)
    pattern = [(-5.5, -4.5), (-1.1, -0.9), (-0.02, 0.0), (-0.02, 0.0), (-5.5, -4.5), (-1.1, -0.9)]
    g = np.empty((T, H, K))
    t = 0
    for s, L in enumerate(lens):
        for c0 in range(0, L, 64):
            lo, hi = pattern[(c0 // 64 + s) % len(pattern)]
            n = min(64, L - c0)
            g[t + c0:t + c0 + n] = rng.uniform(lo, hi, (n, H, K))
        t += L
    d["g"][:T] = inputs.encode16(g)
    og, gg = gates(d, H=H, given_decay=True)
    o, o_ref, s, s_ref, inter, inter_ref = _run(d, H, og, gg)
    assert_o_close(o, o_ref)
    assert_s_close(s, s_ref, "final state")
    assert_s_close(inter, inter_ref, "chunk-start states")


def test_tiny_map_is_applied_to_a_large_state():
    """Decays of about -1 per token make every whole chunk's map about e^-64
    (~5e-28) in size: left out next to states of order B_c (~1e-10), but not
    next to an initial state of order 1e17, where M_c S (~1e-10) outweighs
    B_c.  A skip there would leave most of the second chunk-start state out.
    The ragged last chunk (10 tokens) keeps about e^-10 of its start state,
    so its product runs again."""
    H, lens = 2, [4 * 64 + 10]
    T = sum(lens)
    d = inputs.prefill_inputs(seed=340, lengths=lens, H=H, slots=3)
    rng = np.random.default_rng(341)
    d["g"][:T] = inputs.encode16(rng.uniform(-1.1, -0.9, (T, H, K)))
    d["v"] = inputs.encode16(1e-10 * rng.standard_normal(d["v"].shape))
    d["pool"] = (1e17 * rng.standard_normal(d["pool"].shape)).astype(np.float32)
    og, gg = gates(d, H=H, given_decay=True)
    o, o_ref, s, s_ref, inter, inter_ref = _run(d, H, og, gg)
    assert_s_close(s, s_ref, "final state")
    for c in range(1, inter_ref.shape[0]):  # each chunk-start state on its own scale
        assert_s_close(inter[c], inter_ref[c], f"chunk-start state {c}")
    # outputs from the second chunk on, where the state is of order B_c (the
    # first chunk's outputs are products with the 1e17 state itself)
    assert_o_close(o[64:], o_ref[64:])
