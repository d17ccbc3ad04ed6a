"""GPU parity of the fold's optional branches and of slow decay, through the
C ABI, against the FP64 oracle.

The fold flags follow chunk_kda and the packed-decode validator in "PR #35197
report: fix(kernel) Fix Helion small-token prefill bug" (key source snippets
of kda_prefill.py and kda_decode.py: use_qk_l2norm_in_kernel, A_log, dt_bias,
lower_bound) and beta_is_raw in "[KDA] Support Helion MTP verification and
harden prefill, decode" (sglang PR #42857, Modifications).  Each branch runs
through prefill, decode and chain/tree verify:
  * A_log absent: the gate input is the log-decay itself;
  * beta_is_raw = 0: beta is given in [0, 1];
  * use_qk_l2norm = 0: q and k are drawn with unit-order norms (raw N(0, 1)
    keys of norm ~11 make the update unstable by definition);
  * bounded gates with lower bounds -1 and -5.5 (the chunk form's limit);
    below it, -8, the prefill runs token by token.
Slow decay is where the prefill's state pass carries information over many
chunks, and where its precision matters: full-size prefills at 16 heads with
log-decays in [-0.02, 0] (given) or a bounded gate whose argument is pushed
far negative (g ~ -5 e^-12).  Given log-decays outside the chunk form's
range flag their sequence, which is then computed token by token.
"""
import numpy as np
import pytest
import torch

from linear_attention_serving_gated_gb300 import inputs, kda
from oracle import kda_oracle as ko
from tests.gpu_util import assert_o_close, assert_s_close, dev, dev_bf16, gates

pytestmark = pytest.mark.gpu

K = 128


def _unit_order(x, rng_seed):
    """BF16 N(0, 1/K) values: vectors of norm ~1 for the unnormalised path."""
    rng = np.random.default_rng(rng_seed)
    return inputs.encode16(rng.standard_normal(x.shape).astype(np.float32) * np.float32(K ** -0.5))


def _apply_branch(d, branch, T, tensors):
    """Rewrites seeded inputs in place for one fold branch.  tensors: names of
    (q, k, gate input, beta) in d; T: real token rows of the gate/beta tensors."""
    qn, kn, gn, bn = tensors
    rng = np.random.default_rng(1234)
    if branch == "given_decay":
        d[gn][:T] = inputs.encode16(-rng.uniform(0.0, 5.5, d[gn][:T].shape))
    elif branch == "beta_given":
        d[bn][:T] = inputs.encode16(rng.uniform(0.0, 1.0, d[bn][:T].shape))
    elif branch == "no_l2norm":
        d[qn] = _unit_order(d[qn], 5)
        d[kn] = _unit_order(d[kn], 6)


BRANCHES = {  # name -> gate options
    "given_decay": dict(given_decay=True),
    "beta_given": dict(beta_is_raw=False),
    "no_l2norm": dict(use_qk_l2norm=False),
    "lower_bound_-1": dict(lower_bound=-1.0),
    "lower_bound_-5.5": dict(lower_bound=-5.5),
}


def _prefill(d, H, og, gg, intermediate=True):
    lens = d["lengths"]
    T = int(lens.sum())
    x = {n: dev_bf16(d[n]) for n in ("q", "k", "v", "g", "beta")}
    pool = dev(d["pool"])
    before = pool.clone()
    o = torch.full((T, H, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    nch = int(sum((int(L) + 63) // 64 for L in lens))
    inter = torch.full((nch, H, K, K), float("nan"), device="cuda") if intermediate else None
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_prefill(kda.dims(H), gg, x["q"], x["k"], x["v"], x["g"], x["beta"], pool, dev(d["state_idx"]),
                    dev(d["cu_seqlens"]), len(lens), o, inter, err_flag=err)
    torch.cuda.synchronize()
    opool = d["pool"].astype(np.float64)
    res = ko.prefill(og, d["q"], d["k"], d["v"], d["g"], d["beta"], opool, d["state_idx"], d["cu_seqlens"],
                     intermediate=intermediate)
    o_ref, inter_ref = res if intermediate else (res, None)
    return dict(o=o, pool=pool, before=before, inter=inter, err=int(err.item()), o_ref=o_ref,
                pool_ref=opool, inter_ref=inter_ref)


def _check_prefill(r, d):
    assert r["err"] == 0, f"device error bits {r['err']}"
    worst_o = assert_o_close(r["o"], r["o_ref"])
    slots = [int(s) for s in d["state_idx"] if s >= 0]
    worst_s = assert_s_close(r["pool"][slots], r["pool_ref"][slots], "final state")
    others = [s for s in range(r["pool"].shape[0]) if s not in slots]
    if others:
        assert torch.equal(r["pool"][others], r["before"][others])
    if r["inter"] is not None:  # records of padding sequences (slot -1) are not written
        rows, base = [], 0
        for L, slot in zip(d["lengths"], d["state_idx"]):
            nch = (int(L) + 63) // 64
            if slot >= 0:
                rows.extend(range(base, base + nch))
            base += nch
        worst_s = max(worst_s, assert_s_close(r["inter"][rows], r["inter_ref"][rows], "chunk-start states"))
    return worst_o, worst_s


@pytest.mark.parametrize("branch", sorted(BRANCHES))
def test_prefill_fold_branches(branch):
    H, lens = 4, [1, 63, 64, 65, 200, 130]
    T = sum(lens)
    d = inputs.prefill_inputs(seed=300, lengths=lens, H=H, slots=9, gb_rows=T + 20)
    _apply_branch(d, branch, T, ("q", "k", "g", "beta"))
    og, gg = gates(d, H=H, **BRANCHES[branch])
    _check_prefill(_prefill(d, H, og, gg), d)


@pytest.mark.parametrize("branch", sorted(BRANCHES))
def test_decode_and_verify_fold_branches(branch):
    H, B, T = 4, 5, 6
    opts = BRANCHES[branch]
    D = kda.dims(H)
    # decode: 20 chained steps
    d = inputs.decode_inputs(seed=301, B=B, H=H, slots=12)
    og, gg = gates(d, H=H, **opts)
    pool = dev(d["pool"])
    opool = d["pool"].astype(np.float64)
    idx = dev(d["state_idx"])
    o = torch.empty((B, H, K), dtype=torch.bfloat16, device="cuda")
    for step in range(20):
        x = inputs.decode_step_rows(301, step, B, H)
        qk = x["mixed_qkv"]
        if branch == "no_l2norm":
            qk[:, :2 * H * K] = _unit_order(qk[:, :2 * H * K], step)
        _apply_branch(x, branch if branch != "no_l2norm" else "", B, (None, None, "a", "b"))
        kda.kda_decode_packed(D, gg, dev_bf16(qk), dev_bf16(x["a"]), dev_bf16(x["b"]), pool, idx, o)
        o_ref = ko.decode(og, qk, x["a"], x["b"], opool, d["state_idx"])
        assert_o_close(o, o_ref, f"decode o at step {step}")
    assert_s_close(pool[d["state_idx"]], opool[d["state_idx"]], "decode state")
    # chain and tree verify
    d = inputs.verify_inputs(seed=302, B=B, T=T, H=H, slots=12)
    if branch == "no_l2norm":
        d["mixed_qkv"][:, :2 * H * K] = _unit_order(d["mixed_qkv"][:, :2 * H * K], 7)
    else:
        _apply_branch(d, branch, B * T, (None, None, "a", "b"))
    og, gg = gates(d, H=H, **opts)
    for tree in (False, True):
        pool = dev(d["pool"])
        o = torch.full((B, T, H, K), float("nan"), dtype=torch.bfloat16, device="cuda")
        snaps = torch.full((B, T, H, K, K), float("nan"), device="cuda")
        x = {n: dev_bf16(d[n]) for n in ("mixed_qkv", "a", "b")}
        if tree:
            kda.kda_verify_tree(D, gg, x["mixed_qkv"], x["a"], x["b"], B, T, dev(d["parent"]), pool,
                                dev(d["state_idx"]), o, snaps)
        else:
            kda.kda_verify_chain(D, gg, x["mixed_qkv"], x["a"], x["b"], B, T, pool, dev(d["state_idx"]),
                                 o, snaps)
        o_ref, s_ref = ko.verify(og, d["mixed_qkv"], d["a"], d["b"], B, T, d["pool"].astype(np.float64),
                                 d["state_idx"], d["parent"] if tree else None)
        torch.cuda.synchronize()
        assert_o_close(o, o_ref, f"verify o (tree={tree})")
        assert_s_close(snaps, s_ref, f"verify snapshots (tree={tree})")


# --- slow decay at full size ----------------------------------------------------

def _slow_inputs(T, seed, mode):
    d = inputs.prefill_inputs(seed=seed, lengths=[T], H=16, slots=16)
    if mode == "given":  # log-decays in [-0.02, 0]
        rng = np.random.default_rng(seed + 1)
        d["g"][:T] = inputs.encode16(-0.02 * rng.random(d["g"][:T].shape))
        return d, dict(given_decay=True)
    # bounded gate pushed far into its slow end: g = -5 sigmoid(e^A_log (a - 12))
    d["dt_bias"] = (d["dt_bias"] - np.float32(12.0)).astype(np.float32)
    return d, {}


@pytest.mark.parametrize("T,mode", [(4096, "given"), (4096, "bounded"), (8192, "given")])
def test_prefill_full_size_slow_decay(T, mode):
    """1 x T at 16 heads where each chunk keeps almost all of its start
    state, so the state pass carries it through every chunk: final state and
    chunk-start states within 1e-3 x RMS, o within 2e-2 x RMS."""
    d, opts = _slow_inputs(T, 400 + T // 1024, mode)
    og, gg = gates(d, H=16, **opts)
    _check_prefill(_prefill(d, 16, og, gg, intermediate=(T == 4096)), d)


def test_prefill_many_sequences_slow_decay():
    """40 sequences of 60-330 tokens at 4 heads with given log-decays in
    [-0.02, 0]: every chain product runs, and with 640 (sequence, head,
    slice) items against the SMs each state-pass CTA runs several of them,
    so its copy rings, state buffers and barrier phases carry on from one
    item to the next through the chain products."""
    rng = np.random.default_rng(420)
    lens = [int(x) for x in rng.integers(60, 331, size=40)]
    T = sum(lens)
    d = inputs.prefill_inputs(seed=421, lengths=lens, H=4, slots=48, gb_rows=T + 9)
    d["g"][:T] = inputs.encode16(-0.02 * rng.random(d["g"][:T].shape))
    og, gg = gates(d, H=4, given_decay=True)
    _check_prefill(_prefill(d, 4, og, gg), d)


# --- the prefill's decay range -------------------------------------------------

def test_given_decay_outside_the_chunk_range_takes_the_token_path():
    """A_log absent: a sequence with a log-decay below -5.5 (here -8) or above
    0 is flagged by the decay check, skipped by the chunk transform and the
    state pass, and computed token by token instead; every sequence then
    matches the oracle, with no error bit."""
    H, lens = 2, [70, 50, 90, 40]
    T = sum(lens)
    d = inputs.prefill_inputs(seed=310, lengths=lens, H=H, slots=6, gb_rows=T + 30)
    rng = np.random.default_rng(311)
    d["g"][:T] = inputs.encode16(-rng.uniform(0.0, 5.5, d["g"][:T].shape))
    d["g"][70 + 17, 1, 5] = inputs.encode16(np.array([-8.0]))[0]    # sequence 1
    d["g"][120 + 89, 0, 127] = inputs.encode16(np.array([0.25]))[0]  # sequence 2 (its last row)
    d["g"][T + 3] = inputs.encode16(np.full((H, K), -50.0))           # padding row: never read
    og, gg = gates(d, H=H, given_decay=True)
    _check_prefill(_prefill(d, H, og, gg), d)
    # the same call at the range's edge (-5.5 and 0 exactly) takes the chunk form
    d["g"][70 + 17, 1, 5] = inputs.encode16(np.array([-5.5]))[0]
    d["g"][120 + 89, 0, 127] = 0
    og, gg = gates(d, H=H, given_decay=True)
    _check_prefill(_prefill(d, H, og, gg), d)


def test_bounded_gate_below_the_chunk_range_takes_the_token_path():
    """A bounded gate with lower_bound -8 (past the chunk form's -5.5): every
    sequence runs token by token -- o, chunk-start states and final states
    against the oracle, with a zero-length sequence (state unchanged) and a
    padding sequence (zero outputs, no state) among them."""
    H, lens = 2, [70, 0, 130, 1, 64, 20]
    T = sum(lens)
    idx = [3, 0, 5, -1, 1, 6]
    d = inputs.prefill_inputs(seed=330, lengths=lens, H=H, slots=8, state_idx=idx, gb_rows=T + 11)
    og, gg = gates(d, H=H, lower_bound=-8.0)
    _check_prefill(_prefill(d, H, og, gg), d)


def test_token_path_chunk_ids_past_1024_and_65535_sequences():
    """The token path numbers its chunk-start records by a prefix sum of the
    sequences' chunk counts, taken 1024 sequences at a time, and launches at
    most 65535 sequences at a time: 66000 sequences, nearly all empty, with
    real ones on both sides of each boundary."""
    n, H = 66000, 2
    lens = np.zeros(n, dtype=np.int64)
    real = {3: 70, 1023: 5, 1024: 64, 1025: 1, 2047: 130, 65534: 65, 65535: 1, 65536: 64, 65999: 10}
    for m, L in real.items():
        lens[m] = L
    idx = np.full(n, -1, dtype=np.int32)
    for j, m in enumerate(sorted(real)):
        idx[m] = j
    idx[4], idx[65537] = 9, 10  # empty sequences with a slot: their states stay as they were
    T = int(lens.sum())
    d = inputs.prefill_inputs(seed=340, lengths=lens, H=H, slots=12, state_idx=idx, gb_rows=T + 3)
    og, gg = gates(d, H=H, lower_bound=-8.0)
    _check_prefill(_prefill(d, H, og, gg), d)


def test_short_intermediate_buffer_is_flagged_not_overrun():
    """The chunk-start state buffer holds fewer records than the call's
    sequences have chunks: the records it holds are written, the rest are
    not (the guard record after the buffer stays untouched), and
    KDA_DEVERR_INTERMEDIATE is set."""
    H, lens = 2, [130, 70]  # 3 + 2 = 5 chunks
    T = sum(lens)
    d = inputs.prefill_inputs(seed=320, lengths=lens, H=H, slots=3)
    og, gg = gates(d, H=H)
    x = {n: dev_bf16(d[n]) for n in ("q", "k", "v", "g", "beta")}
    pool = dev(d["pool"])
    store = torch.full((5, H, K, K), 7.0, device="cuda")
    inter = store[:3]  # room for 3 of the 5 records
    o = torch.empty((T, H, K), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_prefill(kda.dims(H), gg, x["q"], x["k"], x["v"], x["g"], x["beta"], pool, dev(d["state_idx"]),
                    dev(d["cu_seqlens"]), 2, o, inter, err_flag=err)
    torch.cuda.synchronize()
    assert err.item() == kda.KDA_DEVERR_INTERMEDIATE
    assert torch.all(store[3:] == 7.0)
    opool = d["pool"].astype(np.float64)
    o_ref, inter_ref = ko.prefill(og, d["q"], d["k"], d["v"], d["g"], d["beta"], opool, d["state_idx"],
                                  d["cu_seqlens"], intermediate=True)
    assert_s_close(store[:3], inter_ref[:3], "chunk-start states within the buffer")
    assert_o_close(o, o_ref)
    assert_s_close(pool[d["state_idx"]], opool[d["state_idx"]])
