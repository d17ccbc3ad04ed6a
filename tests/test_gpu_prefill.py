"""GPU parity of kda_prefill against the FP64 oracle, through the C ABI.

Contract cases follow "PR #35197 report: fix(kernel) Fix Helion small-token
prefill bug" (implementation steps 1-2 and 4: trimmed gate/beta padding rows,
T = 1 handled without poisoning later shapes, fixed and varlen layouts) and
the microbenchmark shapes of "[KDA] Support Helion MTP verification and harden
prefill, decode" (sglang PR #42857, Speed Tests and Profiling: 1x4096,
1x8192, 2x4096 at 16 heads x 128).
"""
import numpy as np
import pytest
import torch

from linear_attention_serving_gated_gb300 import inputs, kda
from oracle import kda_oracle as ko
from tests.gpu_util import assert_o_close, assert_s_close, dev, dev_bf16, gates, host_f64

pytestmark = pytest.mark.gpu

K = 128


def run_both(d, H, varlen=True, intermediate=False, num_seqs=None, oracle=True, gate_kw=None):
    """Runs the CUDA prefill and the oracle on the same inputs (gate_kw: the
    gate's options, default the pages' bounded gate at -5).
    Returns a dict with device results and oracle results."""
    og, gg = gates(d, H=H, **(gate_kw or {}))
    lens = d["lengths"]
    n = len(lens) if num_seqs is None else num_seqs
    T = int(lens.sum())
    x = {name: dev_bf16(d[name]) for name in ("q", "k", "v", "g", "beta")}
    pool = dev(d["pool"])
    pool_before = pool.clone()
    idx = dev(d["state_idx"])
    cu = dev(d["cu_seqlens"]) if varlen else None
    o = torch.full((T, H, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    nch = int(sum((int(L) + 63) // 64 for L in lens))
    inter = torch.full((nch, H, K, K), float("nan"), device="cuda") if intermediate else None
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_prefill(kda.dims(H), gg, x["q"], x["k"], x["v"], x["g"], x["beta"], pool, idx, cu, n, o,
                    inter, err_flag=err)
    torch.cuda.synchronize()
    out = dict(o=o, pool=pool, pool_before=pool_before, inter=inter, err=int(err.item()))
    if oracle:
        opool = d["pool"].astype(np.float64)
        res = ko.prefill(og, d["q"], d["k"], d["v"], d["g"], d["beta"], opool, d["state_idx"],
                         d["cu_seqlens"] if varlen else None, num_seqs=n, intermediate=intermediate)
        out["o_ref"], out["inter_ref"] = (res if intermediate else (res, None))
        out["pool_ref"] = opool
    return out


def check(out, d):
    assert out["err"] == 0
    assert_o_close(out["o"], out["o_ref"])
    idx = [int(s) for s in d["state_idx"] if s >= 0]
    pool = out["pool"]
    assert_s_close(pool[idx], out["pool_ref"][idx], "final state")
    untouched = [s for s in range(pool.shape[0]) if s not in idx]
    if untouched:
        assert torch.equal(pool[untouched], out["pool_before"][untouched]), "untouched slots changed"
    if out["inter"] is not None:  # records of padding sequences (slot -1) are not written
        rows, base = [], 0
        for L, slot in zip(d["lengths"], d["state_idx"]):
            nch = (int(L) + 63) // 64
            if slot >= 0:
                rows.extend(range(base, base + nch))
            base += nch
        assert_s_close(out["inter"][rows], out["inter_ref"][rows], "chunk-start states")


def test_prefill_small_config_128_tokens_4_heads():
    """1 sequence x 128 tokens, 4 heads, slot 0 of a 4-slot pool."""
    d = inputs.prefill_inputs(seed=0, lengths=[128], H=4, slots=4, state_idx=[0])
    check(run_both(d, 4, intermediate=True), d)


@pytest.mark.parametrize("lengths", [[1], [2], [63], [64], [65], [1, 0, 63, 64, 65, 200, 129]])
def test_prefill_ragged_varlen_with_garbage_padding(lengths):
    T = sum(lengths)
    d = inputs.prefill_inputs(seed=len(lengths) * 7 + T, lengths=lengths, H=2, slots=len(lengths) + 3,
                              gb_rows=T + 37)
    check(run_both(d, 2, intermediate=True), d)


def test_prefill_many_short_sequences():
    """300 sequences of 0-70 tokens (several empty, one padding slot) in one
    call: more sequences than one warp step of the transform's and the
    pass's sequence walks (32 at a time), chunk ids resolved across many
    steps, with chunk-start states."""
    rng = np.random.default_rng(11)
    lengths = [int(x) for x in rng.integers(0, 71, size=300)]
    lengths[5] = lengths[40] = lengths[299] = 0
    T = sum(lengths)
    idx = list(rng.permutation(320)[:300])
    idx[17] = -1
    d = inputs.prefill_inputs(seed=12, lengths=lengths, H=2, slots=320, state_idx=idx, gb_rows=T + 5)
    check(run_both(d, 2, intermediate=True), d)


def test_prefill_with_no_tokens_leaves_the_pool_unchanged():
    """The empty call: every sequence has length 0 (one of them a padding
    slot).  No transform runs, the state pass returns before it reads any
    workspace, the pool is untouched and nothing is flagged, as in the
    oracle, where a length-0 sequence passes its state through."""
    d = inputs.prefill_inputs(seed=90, lengths=[0, 0], H=2, slots=4, state_idx=[1, -1])
    out = run_both(d, 2)
    assert out["err"] == 0
    assert out["o"].numel() == 0
    assert torch.equal(out["pool"], out["pool_before"])
    assert np.array_equal(out["pool"].cpu().numpy().astype(np.float64), out["pool_ref"])


def test_prefill_fixed_layout_equal_lengths():
    d = inputs.prefill_inputs(seed=21, lengths=[96, 96, 96], H=2, slots=5, varlen=False)
    check(run_both(d, 2, varlen=False), d)


def test_prefill_fixed_layout_token_path():
    """The fixed layout (no cu_seqlens) on the token-by-token path: a bounded
    gate at -8, and given log-decays with one sequence out of range."""
    d = inputs.prefill_inputs(seed=22, lengths=[130, 130, 130], H=2, slots=5, varlen=False)
    check(run_both(d, 2, varlen=False, intermediate=True, gate_kw=dict(lower_bound=-8.0)), d)
    d = inputs.prefill_inputs(seed=23, lengths=[130, 130, 130], H=2, slots=5, varlen=False)
    rng = np.random.default_rng(24)
    d["g"][:] = inputs.encode16(-rng.uniform(0.0, 5.5, d["g"].shape))
    d["g"][130 + 65, 1, 7] = inputs.encode16(np.array([-9.0]))[0]  # sequence 1 only
    check(run_both(d, 2, varlen=False, intermediate=True, gate_kw=dict(given_decay=True)), d)


def test_single_token_prefill_does_not_poison_later_shapes():
    for seed, lens in ((30, [1]), (31, [130]), (32, [1]), (33, [64, 1, 7])):
        d = inputs.prefill_inputs(seed=seed, lengths=lens, H=2, slots=4, gb_rows=sum(lens) + 5)
        check(run_both(d, 2), d)


@pytest.mark.parametrize("varlen", [True, False])
def test_prefill_ignores_padded_gate_rows(varlen):
    """Same call with NaN/1e4 garbage or zeros in gate/beta padding rows gives
    bitwise-identical results."""
    outs = []
    for garbage in (True, False):
        d = inputs.prefill_inputs(seed=40, lengths=[70, 70], H=2, slots=3, gb_rows=256,
                                  garbage=garbage, varlen=varlen)
        outs.append(run_both(d, 2, varlen=varlen, oracle=garbage))
    check(outs[0], inputs.prefill_inputs(seed=40, lengths=[70, 70], H=2, slots=3, gb_rows=256,
                                         varlen=varlen))
    assert torch.equal(outs[0]["o"], outs[1]["o"])
    assert torch.equal(outs[0]["pool"], outs[1]["pool"])


@pytest.mark.parametrize("T,zero", [(4096, False), (8192, True)])
def test_prefill_full_size_16_heads(T, zero):
    """The pages' single-GPU microbenchmark shape: 1 x T, 16 heads x 128."""
    d = inputs.prefill_inputs(seed=0, lengths=[T], H=16, slots=16, zero_state=zero)
    check(run_both(d, 16), d)


def test_prefill_two_sequences_of_4096():
    d = inputs.prefill_inputs(seed=3, lengths=[4096, 4096], H=16, slots=16, varlen=False)
    check(run_both(d, 16, varlen=False), d)


def test_prefill_varlen_32k_bucket_240_slot_pool():
    """8 sequences U[1,8192] (one of length 1), gate/beta padded to a
    32768-row bucket with garbage, 240-slot pool, random distinct slots."""
    rng = np.random.default_rng(0)
    lens = inputs.varlen_lengths(rng)
    d = inputs.prefill_inputs(seed=0, lengths=lens, H=16, slots=240, gb_rows=32768)
    out = run_both(d, 16)
    check(out, d)


def test_prefill_padding_sequence_and_device_errors():
    d = inputs.prefill_inputs(seed=50, lengths=[40, 33], H=2, slots=4, state_idx=[2, -1])
    out = run_both(d, 2)
    check(out, d)
    assert torch.all(out["o"][40:].float() == 0)
    # out-of-range slot: flagged, sequence skipped, pool untouched
    d = inputs.prefill_inputs(seed=51, lengths=[40, 33], H=2, slots=4, state_idx=[1, 4])
    out = run_both(d, 2, oracle=False)
    assert out["err"] & kda.KDA_DEVERR_SLOT
    assert torch.equal(out["pool"][[0, 2, 3]], out["pool_before"][[0, 2, 3]])
    # malformed cu_seqlens: flagged, nothing written to the pool
    d = inputs.prefill_inputs(seed=52, lengths=[40, 33], H=2, slots=4)
    d["cu_seqlens"] = np.array([0, 80, 73], np.int32)  # ends at T but not non-decreasing
    out = run_both(d, 2, oracle=False)
    assert out["err"] & kda.KDA_DEVERR_SEQLENS
    assert torch.equal(out["pool"], out["pool_before"])


def test_chunked_prefill_across_calls_matches_one_call():
    """Chunked prefill carries state between calls through the pool."""
    d = inputs.prefill_inputs(seed=60, lengths=[150], H=2, slots=3)
    og, gg = gates(d, H=2)
    pool = dev(d["pool"])
    idx = dev(d["state_idx"])
    outs = []
    for a, b in ((0, 90), (90, 150)):
        x = {n: dev_bf16(d[n][a:b]) for n in ("q", "k", "v", "g", "beta")}
        o = torch.empty((b - a, 2, K), dtype=torch.bfloat16, device="cuda")
        kda.kda_prefill(kda.dims(2), gg, x["q"], x["k"], x["v"], x["g"], x["beta"], pool, idx,
                        dev(np.array([0, b - a], np.int32)), 1, o)
        outs.append(o)
    torch.cuda.synchronize()
    opool = d["pool"].astype(np.float64)
    o_ref = ko.prefill(og, d["q"], d["k"], d["v"], d["g"], d["beta"], opool, d["state_idx"],
                       d["cu_seqlens"])
    assert_o_close(torch.cat(outs), o_ref)
    s = int(d["state_idx"][0])
    assert_s_close(pool[s], opool[s])


# --- chains run in two parts ------------------------------------------------
# When 8 * heads * sequences fits the SM count, each (sequence, head) chain of
# chunks runs as two CTAs per value slice; the second restarts behind a chunk
# whose chain product is certainly left out, or from the sequence's start.
# These cases pin long sequences with ragged tails, padding sequences, the
# bit-for-bit agreement with a single CTA per slice, and the dependent launch
# under graph capture.

@pytest.mark.parametrize("T", [16384 + 452, 16385])
def test_long_prefill_in_two_parts_ragged_tail_with_chunk_states(T):
    """1 x T at 2 heads: 264 or 257 chunks in two parts, the last chunk
    ragged (4 tokens, 1 token); chunk-start states too."""
    d = inputs.prefill_inputs(seed=T, lengths=[T], H=2, slots=3, state_idx=[2])
    check(run_both(d, 2, intermediate=True), d)


def test_long_prefill_in_two_parts_fixed_layout_with_padding_sequence():
    d = inputs.prefill_inputs(seed=70, lengths=[16400, 16400], H=2, slots=4, state_idx=[3, -1],
                              varlen=False)
    out = run_both(d, 2, varlen=False)
    check(out, d)
    assert torch.all(out["o"][16400:].float() == 0)


def test_prefill_in_two_parts_bitwise_equals_one_part():
    """Sequence A alone at 16 heads (its chains in two parts) and the same
    tokens as the first sequence of a varlen batch of three (too many chains
    to split: one part each) give identical bits: the split does not change
    the arithmetic."""
    H, TA, TB = 16, 16500, 100
    d = inputs.prefill_inputs(seed=80, lengths=[TA, TB, TB], H=H, slots=4, state_idx=[1, 3, 0])
    og, gg = gates(d, H=H)
    x = {name: dev_bf16(d[name]) for name in ("q", "k", "v", "g", "beta")}
    pool0 = dev(d["pool"])

    pool_a = pool0.clone()
    o_a = torch.zeros((TA, H, K), dtype=torch.bfloat16, device="cuda")
    kda.kda_prefill(kda.dims(H), gg, *(x[n][:TA].contiguous() for n in ("q", "k", "v", "g", "beta")),
                    pool_a, dev(np.array([1], np.int32)), dev(np.array([0, TA], np.int32)), 1, o_a)
    pool_b = pool0.clone()
    o_b = torch.zeros((TA + 2 * TB, H, K), dtype=torch.bfloat16, device="cuda")
    kda.kda_prefill(kda.dims(H), gg, x["q"], x["k"], x["v"], x["g"], x["beta"], pool_b,
                    dev(d["state_idx"]), dev(d["cu_seqlens"]), 3, o_b)
    torch.cuda.synchronize()
    assert torch.equal(o_a, o_b[:TA])
    assert torch.equal(pool_a[1], pool_b[1])


def test_prefill_under_graph_capture_matches_eager():
    """The pass's dependent launch is captured as a programmatic graph
    edge: a replay gives the eager result bit for bit."""
    H, T = 4, 16448
    d = inputs.prefill_inputs(seed=90, lengths=[T], H=H, slots=2, state_idx=[1])
    og, gg = gates(d, H=H)
    x = {name: dev_bf16(d[name]) for name in ("q", "k", "v", "g", "beta")}
    idx, cu = dev(d["state_idx"]), dev(d["cu_seqlens"])
    pool0 = dev(d["pool"])
    ws = torch.empty(kda.kda_prefill_workspace_size(kda.dims(H), 1, T), dtype=torch.uint8, device="cuda")

    pool_e = pool0.clone()
    o_e = torch.empty((T, H, K), dtype=torch.bfloat16, device="cuda")
    kda.kda_prefill(kda.dims(H), gg, x["q"], x["k"], x["v"], x["g"], x["beta"], pool_e, idx, cu, 1, o_e,
                    workspace=ws)
    torch.cuda.synchronize()

    pool_g = pool0.clone()
    o_g = torch.empty_like(o_e)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        kda.kda_prefill(kda.dims(H), gg, x["q"], x["k"], x["v"], x["g"], x["beta"], pool_g, idx, cu, 1,
                        o_g, workspace=ws)
    pool_g.copy_(pool0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o_g, o_e)
    assert torch.equal(pool_g, pool_e)


@pytest.mark.parametrize("given_decay", [False, True])
def test_multi_item_prefill_under_graph_replays_matches_eager(given_decay):
    """More pass items than SMs (300 sequences at 2 heads): the pass's CTAs
    claim items from a workspace counter that each call clears first.
    Replayed twice from a graph (the pool reset between replays), the result
    equals the eager call's bit for bit; with given log-decays the clearing
    is the flags' memset, and one flagged sequence runs token by token."""
    H = 2
    lens = [int(x) for x in np.random.default_rng(91).integers(1, 200, size=300)]
    T = sum(lens)
    d = inputs.prefill_inputs(seed=92, lengths=lens, H=H, slots=310, gb_rows=T + 9)
    if given_decay:
        rng = np.random.default_rng(93)
        d["g"][:T] = inputs.encode16(-rng.uniform(0.0, 5.5, d["g"][:T].shape))
        d["g"][lens[0] + 3, 1, 9] = inputs.encode16(np.array([-7.0]))[0]  # sequence 1
    og, gg = gates(d, H=H, given_decay=given_decay)
    x = {name: dev_bf16(d[name]) for name in ("q", "k", "v", "g", "beta")}
    idx, cu = dev(d["state_idx"]), dev(d["cu_seqlens"])
    pool0 = dev(d["pool"])
    n = len(lens)
    ws = torch.empty(kda.kda_prefill_workspace_size(kda.dims(H), n, T), dtype=torch.uint8, device="cuda")
    pool_e = pool0.clone()
    o_e = torch.empty((T, H, K), dtype=torch.bfloat16, device="cuda")
    kda.kda_prefill(kda.dims(H), gg, x["q"], x["k"], x["v"], x["g"], x["beta"], pool_e, idx, cu, n, o_e,
                    workspace=ws)
    torch.cuda.synchronize()
    opool = d["pool"].astype(np.float64)
    o_ref = ko.prefill(og, d["q"], d["k"], d["v"], d["g"], d["beta"], opool, d["state_idx"], d["cu_seqlens"])
    assert_o_close(o_e, o_ref)

    pool_g = pool0.clone()
    o_g = torch.empty_like(o_e)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        kda.kda_prefill(kda.dims(H), gg, x["q"], x["k"], x["v"], x["g"], x["beta"], pool_g, idx, cu, n,
                        o_g, workspace=ws)
    for _ in range(2):
        pool_g.copy_(pool0)
        o_g.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o_g, o_e)
        assert torch.equal(pool_g, pool_e)
