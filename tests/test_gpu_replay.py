"""GPU parity of the ReplaySSM verify and its commit, through the C ABI.

ReplaySSM is the verify mode the pages measure beside the snapshot mode
("[KDA] Default GLM-5-Next spec verify to the CuTe DSL KDA kernel #42905",
Results: "ReplaySSM rings" against "intermediate-state snapshots"; left out
of the scope of "[KDA] Support Helion MTP verification and harden prefill,
decode", Motivation).  The verify keeps a ring of each draft token's folded
inputs instead of state snapshots, and the commit replays the accepted prefix
onto the pool.  Both are pinned to the snapshot path, which is pinned to the
FP64 oracle elsewhere: outputs and committed states must match it bit for bit,
and the committed states must match the oracle's snapshots within tolerance.
"""
import numpy as np
import pytest
import torch

from linear_attention_serving_gated_gb300 import inputs, kda
from oracle import kda_oracle as ko
from tests.gpu_util import assert_s_close, dev, dev_bf16, gates

pytestmark = pytest.mark.gpu

H, K = 16, 128
D = kda.dims(H)


def _both_paths(d, B, T, gg, accepted):
    x = {n: dev_bf16(d[n]) for n in ("mixed_qkv", "a", "b")}
    idx = dev(d["state_idx"])
    pool_s, pool_r = dev(d["pool"]), dev(d["pool"])
    o_s = torch.full((B, T, H, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    o_r = torch.full_like(o_s, float("nan"))
    snaps = torch.empty((B, T, H, K, K), device="cuda")
    ring = torch.full((kda.kda_replay_ring_bytes(D, B, T) // 4,), float("nan"), device="cuda")
    err = torch.zeros(2, dtype=torch.int32, device="cuda")
    kda.kda_verify_chain(D, gg, x["mixed_qkv"], x["a"], x["b"], B, T, pool_s, idx, o_s, snaps,
                         err_flag=err[0:1])
    before = pool_r.clone()
    kda.kda_verify_chain_replay(D, gg, x["mixed_qkv"], x["a"], x["b"], B, T, pool_r, idx, o_r, ring,
                                err_flag=err[1:2])
    torch.cuda.synchronize()
    assert torch.equal(pool_r, before), "replay verify must not write the pool"
    acc = dev(np.asarray(accepted, np.int32))
    kda.kda_commit(D, snaps, B, T, acc, pool_s, idx, err_flag=err[0:1])
    kda.kda_commit_replay(D, ring, B, T, acc, pool_r, idx, err_flag=err[1:2])
    torch.cuda.synchronize()
    return o_s, o_r, snaps, pool_s, pool_r, [int(e) for e in err.tolist()]


@pytest.mark.parametrize("B", [1, 16, 48])
def test_replay_verify_and_commit_equal_the_snapshot_path(B):
    T = 6
    d = inputs.verify_inputs(seed=300 + B, B=B, T=T, H=H, slots=240)
    og, gg = gates(d, H=H)
    accepted = np.random.default_rng(B).integers(-1, T, size=B)
    o_s, o_r, snaps, pool_s, pool_r, err = _both_paths(d, B, T, gg, accepted)
    assert err == [0, 0]
    assert torch.equal(o_s, o_r), "replay verify outputs differ from the snapshot verify"
    assert torch.equal(pool_s, pool_r), "replayed commit differs from the snapshot commit"
    # and against the oracle's snapshots
    _, s_ref = ko.verify(og, d["mixed_qkv"], d["a"], d["b"], B, T, d["pool"].astype(np.float64),
                         d["state_idx"])
    for r in range(B):
        slot = int(d["state_idx"][r])
        if accepted[r] >= 0:
            assert_s_close(pool_r[slot], s_ref[r, accepted[r]], f"request {r}")
        else:
            assert torch.equal(pool_r[slot], dev(d["pool"])[slot])


def test_replay_longer_than_one_token_block():
    """T = 11 spans two 8-token blocks in the verify and, for the accepted
    indices 8 and 10, in the commit's replay."""
    B, T = 5, 11
    d = inputs.verify_inputs(seed=330, B=B, T=T, H=H, slots=12)
    og, gg = gates(d, H=H)
    o_s, o_r, _, pool_s, pool_r, err = _both_paths(d, B, T, gg, [10, 8, 3, -1, 7])
    assert err == [0, 0]
    assert torch.equal(o_s, o_r)
    assert torch.equal(pool_s, pool_r)


def test_replay_commit_flags_bad_accepted_and_skips_padding():
    B, T = 3, 6
    d = inputs.verify_inputs(seed=310, B=B, T=T, H=H, slots=8)
    d["state_idx"][2] = -1  # padding request
    og, gg = gates(d, H=H)
    o_s, o_r, _, pool_s, pool_r, err = _both_paths(d, B, T, gg, [T, 2, 4])
    assert err[0] & kda.KDA_DEVERR_ACCEPTED and err[1] & kda.KDA_DEVERR_ACCEPTED
    assert torch.all(o_r[2].float() == 0)
    assert torch.equal(o_s, o_r)
    assert torch.equal(pool_s, pool_r)
    assert torch.equal(pool_r[int(d["state_idx"][0])], dev(d["pool"])[int(d["state_idx"][0])])


def test_replay_two_rounds_under_graph_replay():
    """Verify, commit a partial prefix, then change the inputs and slots and
    replay the same CUDA graph: every round equals the eager snapshot path."""
    B, T = 8, 6
    rounds = [inputs.verify_inputs(seed=320 + i, B=B, T=T, H=H, slots=40) for i in range(2)]
    og, gg = gates(rounds[0], H=H)
    pool = dev(rounds[0]["pool"])
    x = {n: dev_bf16(rounds[0][n]) for n in ("mixed_qkv", "a", "b")}
    idx = dev(rounds[0]["state_idx"])
    acc = dev(np.array([5, 0, 3, -1, 2, 5, 1, 4], np.int32))
    o = torch.empty((B, T, H, K), dtype=torch.bfloat16, device="cuda")
    ring = torch.empty((kda.kda_replay_ring_bytes(D, B, T) // 4,), device="cuda")
    kda.kda_verify_chain_replay(D, gg, x["mixed_qkv"], x["a"], x["b"], B, T, pool, idx, o, ring)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        kda.kda_verify_chain_replay(D, gg, x["mixed_qkv"], x["a"], x["b"], B, T, pool, idx, o, ring)
        kda.kda_commit_replay(D, ring, B, T, acc, pool, idx)
    # reference: the snapshot path, eager, on its own pool
    ref_pool = dev(rounds[0]["pool"])
    pool.copy_(ref_pool)
    for i, d in enumerate(rounds):
        for n in ("mixed_qkv", "a", "b"):
            x[n].copy_(dev_bf16(d[n]))
        idx.copy_(dev(d["state_idx"]))
        g.replay()
        snaps = torch.empty((B, T, H, K, K), device="cuda")
        o_ref = torch.empty_like(o)
        kda.kda_verify_chain(D, gg, x["mixed_qkv"], x["a"], x["b"], B, T, ref_pool, idx, o_ref, snaps)
        kda.kda_commit(D, snaps, B, T, acc, ref_pool, idx)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref), f"round {i}: outputs"
        assert torch.equal(pool, ref_pool), f"round {i}: pool"
