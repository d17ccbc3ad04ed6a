"""GPU parity with grouped value heads (HV a multiple of H), through the C ABI.

Value head h reads q/k head h / (HV / H); its v, gate input, beta, gate
parameters and state are its own.  The pages' packed-decode validator ("PR
#35197 report: fix(kernel) Fix Helion small-token prefill bug", kda_decode.py
snippet) takes HV from the state shape and checks the gate input against
HV*K while the q and k widths of a packed row follow H; the oracle follows
the same reading and is pinned to its plain H == HV path (repeated q/k heads).
Every phase is checked against the oracle: prefill (varlen, and a long single
sequence whose chains run in two parts), decode, chain and tree verify with
snapshots, their commit, and the ReplaySSM verify and commit.
"""
import numpy as np
import pytest
import torch

from linear_attention_serving_gated_gb300 import inputs, kda
from oracle import kda_oracle as ko
from tests.gpu_util import assert_o_close, assert_s_close, dev, dev_bf16, gates

pytestmark = pytest.mark.gpu

K = 128


def _prefill(d, Hq, HV, intermediate=False):
    og, gg = gates(d, H=Hq, HV=HV)
    lens = d["lengths"]
    T, n = int(lens.sum()), len(lens)
    x = {name: dev_bf16(d[name]) for name in ("q", "k", "v", "g", "beta")}
    pool = dev(d["pool"])
    nch = int(sum((int(L) + 63) // 64 for L in lens))
    o = torch.full((T, HV, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    inter = torch.full((nch, HV, K, K), float("nan"), device="cuda") if intermediate else None
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_prefill(kda.dims(Hq, HV=HV), gg, x["q"], x["k"], x["v"], x["g"], x["beta"], pool,
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


def test_grouped_prefill_varlen_with_chunk_states():
    d = inputs.prefill_inputs(seed=501, lengths=[1, 63, 200, 65], H=2, HV=4, slots=6, gb_rows=340)
    _prefill(d, 2, 4, intermediate=True)


def test_grouped_prefill_long_single_sequence():
    """16450 tokens (258 chunks) at 4 value heads, the chains in two parts."""
    d = inputs.prefill_inputs(seed=502, lengths=[16450], H=1, HV=4, slots=3, state_idx=[2])
    _prefill(d, 1, 4)


def test_grouped_decode():
    Hq, HV, B = 2, 8, 5
    d = inputs.decode_inputs(seed=503, B=B, H=Hq, HV=HV, slots=9)
    og, gg = gates(d, H=Hq, HV=HV)
    pool = dev(d["pool"])
    o = torch.empty((B, HV, K), dtype=torch.bfloat16, device="cuda")
    kda.kda_decode_packed(kda.dims(Hq, HV=HV), gg, dev_bf16(d["mixed_qkv"]), dev_bf16(d["a"]),
                          dev_bf16(d["b"]), pool, dev(d["state_idx"]), o)
    torch.cuda.synchronize()
    opool = d["pool"].astype(np.float64)
    o_ref = ko.decode(og, d["mixed_qkv"], d["a"], d["b"], opool, d["state_idx"])
    assert_o_close(o, o_ref)
    assert_s_close(pool[d["state_idx"]], opool[d["state_idx"]])


@pytest.mark.parametrize("tree", [False, True])
def test_grouped_verify_and_commit(tree):
    Hq, HV, B, T = 4, 8, 6, 6
    D = kda.dims(Hq, HV=HV)
    d = inputs.verify_inputs(seed=504 + tree, B=B, T=T, H=Hq, HV=HV, slots=11)
    og, gg = gates(d, H=Hq, HV=HV)
    x = {n: dev_bf16(d[n]) for n in ("mixed_qkv", "a", "b")}
    pool, idx = dev(d["pool"]), dev(d["state_idx"])
    o = torch.full((B, T, HV, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    snaps = torch.full((B, T, HV, K, K), float("nan"), device="cuda")
    if tree:
        kda.kda_verify_tree(D, gg, x["mixed_qkv"], x["a"], x["b"], B, T, dev(d["parent"]), pool, idx, o, snaps)
    else:
        kda.kda_verify_chain(D, gg, x["mixed_qkv"], x["a"], x["b"], B, T, pool, idx, o, snaps)
    accepted = np.array([0, 5, -1, 2, 3, 1], np.int32)
    kda.kda_commit(D, snaps, B, T, dev(accepted), pool, idx)
    torch.cuda.synchronize()
    opool = d["pool"].astype(np.float64)
    o_ref, s_ref = ko.verify(og, d["mixed_qkv"], d["a"], d["b"], B, T, opool, d["state_idx"],
                             parent=d["parent"] if tree else None)
    assert_o_close(o, o_ref)
    assert_s_close(snaps, s_ref, "snapshots")
    ko.commit(s_ref, accepted, opool, d["state_idx"])
    assert_s_close(pool[d["state_idx"]], opool[d["state_idx"]], "committed states")


def test_grouped_replay_verify_and_commit_equal_the_snapshot_path():
    Hq, HV, B, T = 2, 4, 7, 6
    D = kda.dims(Hq, HV=HV)
    d = inputs.verify_inputs(seed=506, B=B, T=T, H=Hq, HV=HV, slots=9)
    og, gg = gates(d, H=Hq, HV=HV)
    x = {n: dev_bf16(d[n]) for n in ("mixed_qkv", "a", "b")}
    idx = dev(d["state_idx"])
    pool_s, pool_r = dev(d["pool"]), dev(d["pool"])
    o_s = torch.full((B, T, HV, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    o_r = torch.full_like(o_s, float("nan"))
    snaps = torch.empty((B, T, HV, K, K), device="cuda")
    ring = torch.full((kda.kda_replay_ring_bytes(D, B, T) // 4,), float("nan"), device="cuda")
    kda.kda_verify_chain(D, gg, x["mixed_qkv"], x["a"], x["b"], B, T, pool_s, idx, o_s, snaps)
    kda.kda_verify_chain_replay(D, gg, x["mixed_qkv"], x["a"], x["b"], B, T, pool_r, idx, o_r, ring)
    accepted = dev(np.array([5, 0, -1, 3, 2, 4, 1], np.int32))
    kda.kda_commit(D, snaps, B, T, accepted, pool_s, idx)
    kda.kda_commit_replay(D, ring, B, T, accepted, pool_r, idx)
    torch.cuda.synchronize()
    assert torch.equal(o_s, o_r)
    assert torch.equal(pool_s, pool_r)
