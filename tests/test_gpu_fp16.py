"""GPU parity with FP16 token tensors, through the C ABI.

The pages' prefill sweep covers two precisions ("PR #35197 report:
fix(kernel) Fix Helion small-token prefill bug", implementation step 4)
without naming them; this library reads them as BF16 and FP16 for the token
tensors (q, k, v, gate input, beta, packed rows) and the output o, with FP32
states either way (kda_dims.dtype).  Every phase is checked against the FP64
oracle on the same FP16 inputs, with the same tolerances as BF16 (FP16's own
output rounding, 2^-11 relative, is inside the 2^-8 allowance).
"""
import numpy as np
import pytest
import torch

from linear_attention_serving_gated_gb300 import inputs, kda
from oracle import kda_oracle as ko
from tests.gpu_util import assert_o_close, assert_s_close, dev, dev_in, gates

pytestmark = pytest.mark.gpu

K = 128
F16 = kda.KDA_DTYPE_F16


def _prefill(d, Hq, HV, intermediate=False, lower_bound=-5.0):
    og, gg = gates(d, H=Hq, HV=HV, lower_bound=lower_bound)
    lens = d["lengths"]
    T, n = int(lens.sum()), len(lens)
    x = {name: dev_in(d[name]) for name in ("q", "k", "v", "g", "beta")}
    assert x["q"].dtype == torch.float16
    pool = dev(d["pool"])
    nch = int(sum((int(L) + 63) // 64 for L in lens))
    o = torch.full((T, HV, K), float("nan"), dtype=torch.float16, device="cuda")
    inter = torch.full((nch, HV, K, K), float("nan"), device="cuda") if intermediate else None
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_prefill(kda.dims(Hq, HV=HV, dtype=F16), gg, x["q"], x["k"], x["v"], x["g"], x["beta"], pool,
                    dev(d["state_idx"]), dev(d["cu_seqlens"]), n, o, inter, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    opool = d["pool"].astype(np.float64)
    res = ko.prefill(og, d["q"], d["k"], d["v"], d["g"], d["beta"], opool, d["state_idx"], d["cu_seqlens"],
                     intermediate=intermediate)
    o_ref, inter_ref = res if intermediate else (res, None)
    assert_o_close(o, o_ref)
    idx = [int(s) for s in d["state_idx"] if s >= 0]
    assert_s_close(pool[idx], opool[idx], "final state")
    if intermediate:
        assert_s_close(inter, inter_ref, "chunk-start states")


def test_fp16_prefill_varlen_with_garbage_padding_and_chunk_states():
    d = inputs.prefill_inputs(seed=601, lengths=[1, 64, 130, 65, 0, 7], H=2, slots=8, gb_rows=300,
                              dtype="f16")
    _prefill(d, 2, 2, intermediate=True)


def test_fp16_prefill_single_sequence_16_heads():
    """1 x 4096 at 16 heads: the benchmark shape."""
    d = inputs.prefill_inputs(seed=602, lengths=[4096], H=16, slots=16, dtype="f16")
    _prefill(d, 16, 16)


def test_fp16_grouped_heads_prefill():
    d = inputs.prefill_inputs(seed=603, lengths=[200, 33], H=2, HV=4, slots=5, dtype="f16")
    _prefill(d, 2, 4)


def test_fp16_grouped_heads_prefill_token_path():
    """A bounded gate below the chunk form's range (lower_bound -8): every
    sequence runs token by token, here with FP16 rows and two value heads
    per q/k head."""
    d = inputs.prefill_inputs(seed=604, lengths=[130, 1, 64, 70], H=2, HV=4, slots=6, gb_rows=280, dtype="f16")
    _prefill(d, 2, 4, intermediate=True, lower_bound=-8.0)


def test_fp16_decode_chained_steps():
    H, B = 16, 16
    D = kda.dims(H, dtype=F16)
    d = inputs.decode_inputs(seed=604, B=B, H=H, slots=40, dtype="f16")
    og, gg = gates(d, H=H)
    pool = dev(d["pool"])
    opool = d["pool"].astype(np.float64)
    idx = dev(d["state_idx"])
    o = torch.empty((B, H, K), dtype=torch.float16, device="cuda")
    for step in range(50):
        x = inputs.decode_step_rows(604, step, B, H, dtype="f16")
        kda.kda_decode_packed(D, gg, dev_in(x["mixed_qkv"]), dev_in(x["a"]), dev_in(x["b"]), pool, idx, o)
        o_ref = ko.decode(og, x["mixed_qkv"], x["a"], x["b"], opool, d["state_idx"])
        assert_o_close(o, o_ref, f"o at step {step}")
    assert_s_close(pool[d["state_idx"]], opool[d["state_idx"]])


@pytest.mark.parametrize("tree", [False, True])
def test_fp16_verify_and_commit(tree):
    H, B, T = 16, 12, 6
    D = kda.dims(H, dtype=F16)
    d = inputs.verify_inputs(seed=605 + tree, B=B, T=T, H=H, slots=30, dtype="f16")
    og, gg = gates(d, H=H)
    x = {n: dev_in(d[n]) for n in ("mixed_qkv", "a", "b")}
    pool, idx = dev(d["pool"]), dev(d["state_idx"])
    o = torch.full((B, T, H, K), float("nan"), dtype=torch.float16, device="cuda")
    snaps = torch.full((B, T, H, K, K), float("nan"), device="cuda")
    if tree:
        kda.kda_verify_tree(D, gg, x["mixed_qkv"], x["a"], x["b"], B, T, dev(d["parent"]), pool, idx, o, snaps)
    else:
        kda.kda_verify_chain(D, gg, x["mixed_qkv"], x["a"], x["b"], B, T, pool, idx, o, snaps)
    accepted = np.random.default_rng(605).integers(-1, T, size=B).astype(np.int32)
    kda.kda_commit(D, snaps, B, T, dev(accepted), pool, idx)
    torch.cuda.synchronize()
    opool = d["pool"].astype(np.float64)
    o_ref, s_ref = ko.verify(og, d["mixed_qkv"], d["a"], d["b"], B, T, opool, d["state_idx"],
                             parent=d["parent"] if tree else None)
    assert_o_close(o, o_ref)
    assert_s_close(snaps, s_ref, "snapshots")
    ko.commit(s_ref, accepted, opool, d["state_idx"])
    assert_s_close(pool[d["state_idx"]], opool[d["state_idx"]], "committed states")


def test_fp16_replay_verify_and_commit_equal_the_snapshot_path():
    H, B, T = 16, 5, 6
    D = kda.dims(H, dtype=F16)
    d = inputs.verify_inputs(seed=607, B=B, T=T, H=H, slots=20, dtype="f16")
    og, gg = gates(d, H=H)
    x = {n: dev_in(d[n]) for n in ("mixed_qkv", "a", "b")}
    idx = dev(d["state_idx"])
    pool_s, pool_r = dev(d["pool"]), dev(d["pool"])
    o_s = torch.full((B, T, H, K), float("nan"), dtype=torch.float16, device="cuda")
    o_r = torch.full_like(o_s, float("nan"))
    snaps = torch.empty((B, T, H, K, K), device="cuda")
    ring = torch.full((kda.kda_replay_ring_bytes(D, B, T) // 4,), float("nan"), device="cuda")
    kda.kda_verify_chain(D, gg, x["mixed_qkv"], x["a"], x["b"], B, T, pool_s, idx, o_s, snaps)
    kda.kda_verify_chain_replay(D, gg, x["mixed_qkv"], x["a"], x["b"], B, T, pool_r, idx, o_r, ring)
    accepted = dev(np.array([5, 0, -1, 3, 2], np.int32))
    kda.kda_commit(D, snaps, B, T, accepted, pool_s, idx)
    kda.kda_commit_replay(D, ring, B, T, accepted, pool_r, idx)
    torch.cuda.synchronize()
    assert torch.equal(o_s, o_r)
    assert torch.equal(pool_s, pool_r)


def test_dtype_mismatch_is_refused_by_the_binding():
    d = inputs.decode_inputs(seed=608, B=2, H=2, slots=4, dtype="f16")
    og, gg = gates(d, H=2)
    o = torch.empty((2, 2, K), dtype=torch.float16, device="cuda")
    with pytest.raises(TypeError):  # FP16 tensors under a BF16 dims
        kda.kda_decode_packed(kda.dims(2), gg, dev_in(d["mixed_qkv"]), dev_in(d["a"]), dev_in(d["b"]),
                              dev(d["pool"]), dev(d["state_idx"]), o)
