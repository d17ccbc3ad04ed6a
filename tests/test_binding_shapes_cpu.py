"""Host-side shape rules of the Python binding, which the C ABI cannot see
(it takes pointers).  The packed-row rules follow the pages' packed-decode
validator ("PR #35197 report: fix(kernel) Fix Helion small-token prefill
bug", kda_decode.py snippet): HV, V and K come from the state's trailing
dimensions and the gate input must be [B, HV*K].  The others keep every row
a kernel touches inside its buffer.

CPU tensors are used: the shape checks run before the pointers are taken,
so a well-shaped call gets as far as the device-tensor check and no further.
"""
import pytest
import torch

from linear_attention_serving_gated_gb300 import build, kda

H, K = 2, 128
BF = torch.bfloat16


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return kda.load()


def rows(n, H=H, HV=H):
    return dict(mixed_qkv=torch.zeros((n, 2 * H * K + HV * K), dtype=BF),
                a=torch.zeros((n, HV * K), dtype=BF), b=torch.zeros((n, HV), dtype=BF))


def pool(HV=H, slots=4):
    return torch.zeros((slots, HV, K, K))


def idx(n):
    return torch.zeros(n, dtype=torch.int32)


def decode(x, p=None, o=None, d=None, B=2):
    kda.kda_decode_packed(d or kda.dims(H), kda.Gate(), x["mixed_qkv"], x["a"], x["b"],
                          pool() if p is None else p, idx(B),
                          torch.zeros((B, H, K), dtype=BF) if o is None else o)


def test_well_shaped_decode_reaches_the_pointer_check():
    with pytest.raises(ValueError, match="device tensors"):
        decode(rows(2))


def test_gate_input_must_be_B_by_HV_K():
    x = rows(2)
    x["a"] = torch.zeros((2, H * K - 8), dtype=BF)
    with pytest.raises(ValueError, match="`a` must have shape"):
        decode(x)
    x["a"] = torch.zeros((2, 2 * H * K), dtype=BF)[:, ::2]  # right shape, not contiguous
    with pytest.raises(ValueError, match="`a` must have shape"):
        decode(x)


def test_state_pool_gives_HV_V_K():
    with pytest.raises(ValueError, match="state_pool must end in"):
        decode(rows(2), p=torch.zeros((4, H + 1, K, K)))
    with pytest.raises(ValueError, match="state_pool must end in"):
        decode(rows(2), p=torch.zeros((4, H, K, 64)))


def test_grouped_heads_widths():
    d = kda.dims(2, HV=4)
    x = rows(2, H=2, HV=4)
    o = torch.zeros((2, 4, K), dtype=BF)
    with pytest.raises(ValueError, match="device tensors"):
        decode(x, p=pool(HV=4), o=o, d=d)
    x["b"] = torch.zeros((2, 2), dtype=BF)  # beta per q/k head instead of per value head
    with pytest.raises(ValueError, match="`b` must have shape"):
        decode(x, p=pool(HV=4), o=o, d=d)


def test_decode_output_must_hold_every_row():
    with pytest.raises(ValueError, match="o must hold"):
        decode(rows(2), o=torch.zeros((1, H, K), dtype=BF))


def test_buffers_must_be_dense():
    """The library indexes every buffer by its documented dense layout (only
    mixed_qkv carries a row stride)."""
    with pytest.raises(ValueError, match="o must be contiguous"):
        decode(rows(2), o=torch.zeros((H, 2, K), dtype=BF).transpose(0, 1))
    with pytest.raises(ValueError, match="state_pool must be contiguous"):
        decode(rows(2), p=torch.zeros((4, K, K, H)).permute(0, 3, 1, 2))
    x = rows(2)
    x["mixed_qkv"] = torch.zeros((2, 2 * (2 * H * K + H * K)), dtype=BF)[:, :2 * H * K + H * K]
    with pytest.raises(ValueError, match="device tensors"):  # a row stride is fine for mixed_qkv
        decode(x)


def verify(B, T, x, snaps=None, o=None, parent=None, tree=False):
    o = torch.zeros((B, T, H, K), dtype=BF) if o is None else o
    snaps = torch.zeros((B, T, H, K, K)) if snaps is None else snaps
    if tree:
        kda.kda_verify_tree(kda.dims(H), kda.Gate(), x["mixed_qkv"], x["a"], x["b"], B, T,
                            torch.zeros(B * T, dtype=torch.int32) if parent is None else parent,
                            pool(), idx(B), o, snaps)
    else:
        kda.kda_verify_chain(kda.dims(H), kda.Gate(), x["mixed_qkv"], x["a"], x["b"], B, T,
                             pool(), idx(B), o, snaps)


def test_verify_reads_B_times_T_rows():
    with pytest.raises(ValueError, match="device tensors"):
        verify(2, 3, rows(6))
    with pytest.raises(ValueError, match="mixed_qkv must be"):
        verify(2, 3, rows(5))


def test_verify_outputs_and_parents_must_hold_every_token():
    with pytest.raises(ValueError, match="snapshots must hold"):
        verify(2, 3, rows(6), snaps=torch.zeros((2, 2, H, K, K)))
    with pytest.raises(ValueError, match="o must hold"):
        verify(2, 3, rows(6), o=torch.zeros((2, 2, H, K), dtype=BF))
    with pytest.raises(ValueError, match="parent_idx must hold"):
        verify(2, 3, rows(6), parent=torch.zeros(5, dtype=torch.int32), tree=True)


def test_replay_ring_and_commits():
    B, T = 2, 3
    x = rows(B * T)
    d = kda.dims(H)
    short_ring = torch.zeros(kda.kda_replay_ring_bytes(d, B, T) // 4 - 1)
    with pytest.raises(ValueError, match="ring must hold"):
        kda.kda_verify_chain_replay(d, kda.Gate(), x["mixed_qkv"], x["a"], x["b"], B, T, pool(),
                                    idx(B), torch.zeros((B, T, H, K), dtype=BF), short_ring)
    with pytest.raises(ValueError, match="ring must hold"):
        kda.kda_commit_replay(d, short_ring, B, T, idx(B), pool(), idx(B))
    with pytest.raises(ValueError, match="accepted must hold"):
        kda.kda_commit(d, torch.zeros((B, T, H, K, K)), B, T, idx(B - 1), pool(), idx(B))
    with pytest.raises(ValueError, match="state_idx must hold"):
        kda.kda_commit(d, torch.zeros((B, T, H, K, K)), B, T, idx(B), pool(), idx(B - 1))


def prefill(T=100, o=None, n=1, cu_len=None, idx_len=None, inter=None):
    q = torch.zeros((T, H, K), dtype=BF)
    kda.kda_prefill(kda.dims(H), kda.Gate(), q, q.clone(), q.clone(), torch.zeros((T, H, K), dtype=BF),
                    torch.zeros((T, H), dtype=BF), pool(), idx(n if idx_len is None else idx_len),
                    torch.zeros(n + 1 if cu_len is None else cu_len, dtype=torch.int32), n,
                    torch.zeros((T, H, K), dtype=BF) if o is None else o, inter,
                    workspace=torch.zeros(16, dtype=torch.uint8))


def test_prefill_intermediate_is_a_stack_of_state_records():
    """The chunk-start state buffer's record count is passed to the library
    (which writes no more than that many), so it must be a dense float32
    [chunks, HV, V, K] tensor."""
    for bad in (torch.zeros((2, H, K, K - 1)), torch.zeros((2, H, K, K), dtype=torch.float64),
                torch.zeros((2 * H * K * K,)), torch.zeros((2, K, K, H)).permute(0, 3, 1, 2)):
        with pytest.raises(ValueError, match="intermediate must be"):
            prefill(inter=bad)


def test_prefill_shapes():
    with pytest.raises(ValueError, match="device tensors"):
        prefill()
    with pytest.raises(ValueError, match="o must hold"):
        prefill(o=torch.zeros((99, H, K), dtype=BF))
    with pytest.raises(ValueError, match="cu_seqlens must hold"):
        prefill(n=2, cu_len=2)
    with pytest.raises(ValueError, match="state_idx must hold"):
        prefill(n=2, idx_len=1)
