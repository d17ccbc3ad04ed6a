"""GPU parity of packed decode, chain/tree verify and commit against the
FP64 oracle, through the C ABI.

Cases follow "[KDA] Support Helion MTP verification and harden prefill,
decode" (sglang PR #42857): packed decode at 1/16/48 requests, verify with
per-candidate state snapshots at 6 draft tokens, chain and tree, and the
review thread's two-round contract (verify, commit a partially accepted
prefix, change inputs and slot indices, replay the same CUDA graph); the
GB300 request sweep 1..48 of "[KDA] Default GLM-5-Next spec verify to the
CuTe DSL KDA kernel" (#42905, Results); the decode input contract of
validate_packed_decode_inputs ("PR #35197 report", kda_decode.py snippet).
"""
import numpy as np
import pytest
import torch

from linear_attention_serving_gated_gb300 import inputs, kda
from oracle import kda_oracle as ko
from tests.gpu_util import assert_o_close, assert_s_close, dev, dev_bf16, gates

pytestmark = pytest.mark.gpu

H, K = 16, 128
D = kda.dims(H)


@pytest.mark.parametrize("B", [1, 16, 48])
def test_decode_1000_chained_steps(B):
    d = inputs.decode_inputs(seed=B, B=B, H=H, slots=240)
    og, gg = gates(d, H=H)
    pool = dev(d["pool"])
    before = pool.clone()
    opool = d["pool"].astype(np.float64)
    idx = dev(d["state_idx"])
    o = torch.empty((B, H, K), dtype=torch.bfloat16, device="cuda")
    steps = 1000
    worst_o = 0.0
    for step in range(steps):
        x = inputs.decode_step_rows(B, step, B, H)
        kda.kda_decode_packed(D, gg, dev_bf16(x["mixed_qkv"]), dev_bf16(x["a"]), dev_bf16(x["b"]),
                              pool, idx, o)
        o_ref = ko.decode(og, x["mixed_qkv"], x["a"], x["b"], opool, d["state_idx"])
        worst_o = max(worst_o, assert_o_close(o, o_ref, f"o at step {step}"))
        if step % 250 == 249:
            assert_s_close(pool[d["state_idx"]], opool[d["state_idx"]], f"state at step {step}")
    untouched = np.setdiff1d(np.arange(240), d["state_idx"])
    assert torch.equal(pool[untouched], before[untouched])


def test_decode_padding_request_and_bad_slot():
    d = inputs.decode_inputs(seed=5, B=4, H=H, slots=8)
    og, gg = gates(d, H=H)
    idx = d["state_idx"].copy()
    idx[1] = -1
    idx[3] = 8  # out of range
    pool = dev(d["pool"])
    before = pool.clone()
    o = torch.full((4, H, K), 7.0, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_decode_packed(D, gg, dev_bf16(d["mixed_qkv"]), dev_bf16(d["a"]), dev_bf16(d["b"]),
                          pool, dev(idx), o, err_flag=err)
    torch.cuda.synchronize()
    assert err.item() & kda.KDA_DEVERR_SLOT
    assert torch.all(o[1].float() == 0) and torch.all(o[3].float() == 0)
    opool = d["pool"].astype(np.float64)
    ok_idx = idx.copy()
    ok_idx[3] = -1
    o_ref = ko.decode(og, d["mixed_qkv"], d["a"], d["b"], opool, ok_idx)
    assert_o_close(o[[0, 2]], o_ref[[0, 2]])
    touched = [int(idx[0]), int(idx[2])]
    assert_s_close(pool[touched], opool[touched])
    untouched = [s for s in range(8) if s not in touched]
    assert torch.equal(pool[untouched], before[untouched])


def test_decode_graph_replay_with_new_indices():
    """Indices and inputs are read on the device at run time, so a captured
    graph replays correctly after they change."""
    B = 16
    d = inputs.decode_inputs(seed=9, B=B, H=H, slots=64)
    og, gg = gates(d, H=H)
    x = {n: dev_bf16(d[n]) for n in ("mixed_qkv", "a", "b")}
    pool = dev(d["pool"])
    idx = dev(d["state_idx"])
    o = torch.empty((B, H, K), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        kda.kda_decode_packed(D, gg, x["mixed_qkv"], x["a"], x["b"], pool, idx, o)  # warm-up
    torch.cuda.current_stream().wait_stream(s)
    pool.copy_(dev(d["pool"]))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        kda.kda_decode_packed(D, gg, x["mixed_qkv"], x["a"], x["b"], pool, idx, o)
    opool = d["pool"].astype(np.float64)
    rng = np.random.default_rng(99)
    for rnd in range(3):
        new_idx = rng.permutation(64)[:B].astype(np.int32)
        rows = inputs.decode_step_rows(9, rnd, B, H)
        idx.copy_(dev(new_idx))
        for n in ("mixed_qkv", "a", "b"):
            x[n].copy_(dev_bf16(rows[n]))
        graph.replay()
        torch.cuda.synchronize()
        o_ref = ko.decode(og, rows["mixed_qkv"], rows["a"], rows["b"], opool, new_idx)
        assert_o_close(o, o_ref)
    assert_s_close(pool, opool)


def _verify(d, B, T, tree, og, gg, pool=None):
    x = {n: dev_bf16(d[n]) for n in ("mixed_qkv", "a", "b")}
    pool = dev(d["pool"]) if pool is None else pool
    before = pool.clone()
    idx = dev(d["state_idx"])
    o = torch.full((B, T, H, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    snaps = torch.full((B, T, H, K, K), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if tree:
        kda.kda_verify_tree(D, gg, x["mixed_qkv"], x["a"], x["b"], B, T, dev(d["parent"]), pool, idx,
                            o, snaps, err_flag=err)
    else:
        kda.kda_verify_chain(D, gg, x["mixed_qkv"], x["a"], x["b"], B, T, pool, idx, o, snaps,
                             err_flag=err)
    torch.cuda.synchronize()
    assert torch.equal(pool, before), "verify must not write the pool"
    return o, snaps, int(err.item())


@pytest.mark.parametrize("B", [1, 2, 4, 8, 12, 16, 24, 32, 48])
@pytest.mark.parametrize("tree", [False, True])
def test_verify_six_draft_tokens(B, tree):
    T = 6
    d = inputs.verify_inputs(seed=100 + B, B=B, T=T, H=H, slots=240)
    og, gg = gates(d, H=H)
    o, snaps, err = _verify(d, B, T, tree, og, gg)
    assert err == 0
    opool = d["pool"].astype(np.float64)
    o_ref, s_ref = ko.verify(og, d["mixed_qkv"], d["a"], d["b"], B, T, opool, d["state_idx"],
                             parent=d["parent"] if tree else None)
    assert_o_close(o, o_ref)
    assert_s_close(snaps, s_ref, "snapshots")


def test_tree_with_chain_parents_is_bitwise_chain():
    B, T = 8, 6
    d = inputs.verify_inputs(seed=7, B=B, T=T, H=H, slots=32)
    og, gg = gates(d, H=H)
    oc, sc, _ = _verify(d, B, T, False, og, gg)
    d["parent"] = np.tile(np.arange(-1, T - 1, dtype=np.int32), (B, 1))
    ot, st, _ = _verify(d, B, T, True, og, gg)
    assert torch.equal(oc, ot) and torch.equal(sc, st)


def test_tree_bad_parent_flags_and_skips():
    B, T = 3, 6
    d = inputs.verify_inputs(seed=8, B=B, T=T, H=H, slots=8)
    og, gg = gates(d, H=H)
    d["parent"][1, 3] = 3  # not < 3
    o, snaps, err = _verify(d, B, T, True, og, gg)
    assert err & kda.KDA_DEVERR_PARENT
    assert torch.all(o[1].float() == 0)
    o_ref, s_ref = ko.verify(og, d["mixed_qkv"][[0, 1, 2, 3, 4, 5, 12, 13, 14, 15, 16, 17]],
                             d["a"][[0, 1, 2, 3, 4, 5, 12, 13, 14, 15, 16, 17]],
                             d["b"][[0, 1, 2, 3, 4, 5, 12, 13, 14, 15, 16, 17]], 2, T,
                             d["pool"].astype(np.float64), d["state_idx"][[0, 2]],
                             parent=d["parent"][[0, 2]])
    assert_o_close(o[[0, 2]], o_ref)
    assert_s_close(snaps[[0, 2]], s_ref)


def test_commit_is_bit_exact_and_respects_minus_one():
    B, T = 6, 6
    d = inputs.verify_inputs(seed=11, B=B, T=T, H=H, slots=20)
    og, gg = gates(d, H=H)
    pool = dev(d["pool"])
    o, snaps, _ = _verify(d, B, T, False, og, gg, pool=pool)
    before = pool.clone()
    acc = np.array([0, -1, 5, 2, -1, 3], np.int32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_commit(D, snaps, B, T, dev(acc), pool, dev(d["state_idx"]), err_flag=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    for r in range(B):
        s = int(d["state_idx"][r])
        if acc[r] < 0:
            assert torch.equal(pool[s], before[s])
        else:
            assert torch.equal(pool[s], snaps[r, acc[r]])
    others = np.setdiff1d(np.arange(20), d["state_idx"])
    assert torch.equal(pool[others], before[others])
    acc_bad = np.array([0, 6, -1, -1, -1, -1], np.int32)
    kda.kda_commit(D, snaps, B, T, dev(acc_bad), pool, dev(d["state_idx"]), err_flag=err)
    torch.cuda.synchronize()
    assert err.item() & kda.KDA_DEVERR_ACCEPTED


@pytest.mark.parametrize("tree", [False, True])
def test_two_round_verify_commit_under_graph_replay(tree):
    """Round 1: verify, commit a partially accepted prefix.  Round 2: new
    inputs and new slot indices copied into the captured buffers, the same
    graph replayed.  Outputs and snapshots match the oracle doing the same,
    and the committed states are preserved."""
    B, T, slots = 8, 6, 48
    d1 = inputs.verify_inputs(seed=200, B=B, T=T, H=H, slots=slots)
    og, gg = gates(d1, H=H)
    x = {n: dev_bf16(d1[n]) for n in ("mixed_qkv", "a", "b")}
    par = dev(d1["parent"])
    pool = dev(d1["pool"])
    idx = dev(d1["state_idx"])
    acc = torch.zeros(B, dtype=torch.int32, device="cuda")
    o = torch.empty((B, T, H, K), dtype=torch.bfloat16, device="cuda")
    snaps = torch.empty((B, T, H, K, K), device="cuda")

    def step():
        if tree:
            kda.kda_verify_tree(D, gg, x["mixed_qkv"], x["a"], x["b"], B, T, par, pool, idx, o, snaps)
        else:
            kda.kda_verify_chain(D, gg, x["mixed_qkv"], x["a"], x["b"], B, T, pool, idx, o, snaps)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    opool = d1["pool"].astype(np.float64)
    rng = np.random.default_rng(5)
    d = d1
    for rnd in range(2):
        if rnd == 1:
            d = inputs.verify_inputs(seed=201, B=B, T=T, H=H, slots=slots)
            d["state_idx"] = rng.permutation(slots)[:B].astype(np.int32)
            for n in ("mixed_qkv", "a", "b"):
                x[n].copy_(dev_bf16(d[n]))
            par.copy_(dev(d["parent"]))
            idx.copy_(dev(d["state_idx"]))
        graph.replay()
        torch.cuda.synchronize()
        o_ref, s_ref = ko.verify(og, d["mixed_qkv"], d["a"], d["b"], B, T, opool, d["state_idx"],
                                 parent=d["parent"] if tree else None)
        assert_o_close(o, o_ref, f"o round {rnd}")
        assert_s_close(snaps, s_ref, f"snapshots round {rnd}")
        accepted = rng.integers(-1, T, size=B).astype(np.int32)
        acc.copy_(dev(accepted))
        kda.kda_commit(D, snaps, B, T, acc, pool, idx)
        ko.commit(s_ref, accepted, opool, d["state_idx"])
        torch.cuda.synchronize()
        assert_s_close(pool, opool, f"pool after commit round {rnd}")
