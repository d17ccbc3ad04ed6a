"""C-ABI checks that need no GPU: the library loads, exports every entry
point include/kda.h declares, and rejects bad host-side arguments with the
status codes that mirror the pages' ValueErrors ("PR #35197 report:
fix(kernel) Fix Helion small-token prefill bug", key source snippets of
kda_prefill.py and kda_decode.py).  Every call here returns before touching
the device, so dummy non-NULL pointers are safe."""
import ctypes
import math
import os
import re

import pytest

from linear_attention_serving_gated_gb300 import build, kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")
DUMMY = ctypes.c_void_p(0x10000)  # 16-byte aligned, never dereferenced


@pytest.fixture(scope="module")
def lib():
    build.build()
    return kda.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(kda.EXPORTS), names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for s in range(7):
        assert kda.status_string(s)
    assert "workspace" in kda.status_string(kda.KDA_ERR_WORKSPACE)


REC_BYTES = 180352  # one (chunk, head) record, as include/kda.h states


def test_workspace_size_formula(lib):
    """align256(4 num_seqs + 4) + (T / 64 + num_seqs) HV 180352 + num_seqs HV
    65536 bytes, as kda.h states; sizes past int32 tokens give SIZE_MAX so
    that no check passes."""
    for HV, n, T in ((16, 1, 64), (16, 1, 4096), (16, 8, 32768), (4, 3, 100), (2, 70, 0), (16, 64, 4096)):
        want = ((4 * n + 4 + 255) // 256) * 256 + (T // 64 + n) * HV * REC_BYTES + n * HV * 65536
        assert kda.kda_prefill_workspace_size(kda.dims(HV), n, T) == want
    assert kda.kda_prefill_workspace_size(kda.dims(16), 1, 2 ** 31) == 2 ** 64 - 1
    assert kda.kda_prefill_workspace_size(kda.dims(16), 1, 2 ** 31 - 1) < 2 ** 63


def _gate(A_log=None, lb=-5.0):
    return kda.kda_gate(A_log, None, lb, 1, 1, 128 ** -0.5)


def _prefill(lib, dims=None, gate=None, pool=DUMMY, idx=DUMMY, gb_rows=64, T=64, num_seqs=1,
             ws=DUMMY, ws_bytes=1 << 40, q=DUMMY, inter=None, inter_chunks=0):
    return lib.kda_prefill(dims or kda.dims(4), gate or _gate(), q, DUMMY, DUMMY, DUMMY, DUMMY,
                           gb_rows, pool, 4, idx, None, num_seqs, T, DUMMY, inter, inter_chunks, ws,
                           ws_bytes, None, None)


def test_prefill_host_errors(lib):
    # no pool or no indices: an indexed initial-state pool is required
    assert _prefill(lib, pool=None) == kda.KDA_ERR_NULL_ARG
    assert _prefill(lib, idx=None) == kda.KDA_ERR_NULL_ARG
    # gate/beta must cover every q token
    assert _prefill(lib, gb_rows=63) == kda.KDA_ERR_SHAPE
    # non-power-of-two head dims are rejected; other shapes are not built
    assert _prefill(lib, dims=kda.dims(4, K=96, V=128)) == kda.KDA_ERR_UNSUPPORTED
    assert _prefill(lib, dims=kda.dims(4, K=128, V=100)) == kda.KDA_ERR_UNSUPPORTED
    assert _prefill(lib, dims=kda.dims(4, K=64, V=64)) == kda.KDA_ERR_UNSUPPORTED
    # value heads come in whole groups per q/k head (HV a multiple of H)
    assert _prefill(lib, dims=kda.dims(4, HV=6)) == kda.KDA_ERR_UNSUPPORTED
    assert _prefill(lib, dims=kda.dims(4, HV=2)) == kda.KDA_ERR_UNSUPPORTED
    # token tensors are BF16 or FP16
    assert _prefill(lib, dims=kda.dims(4, dtype=2)) == kda.KDA_ERR_UNSUPPORTED
    # bounded gate formula only
    assert _prefill(lib, gate=_gate(A_log=DUMMY, lb=math.nan)) == kda.KDA_ERR_UNSUPPORTED
    # fixed layout needs equal lengths
    assert _prefill(lib, T=65, gb_rows=65, num_seqs=2) == kda.KDA_ERR_SHAPE
    # workspace
    assert _prefill(lib, ws=None) == kda.KDA_ERR_WORKSPACE
    assert _prefill(lib, ws_bytes=16) == kda.KDA_ERR_WORKSPACE
    assert _prefill(lib, ws=ctypes.c_void_p(0x10010)) == kda.KDA_ERR_ALIGNMENT
    assert _prefill(lib, q=ctypes.c_void_p(0x10002)) == kda.KDA_ERR_ALIGNMENT
    # cu_seqlens are int32: more tokens than that is a shape error
    assert _prefill(lib, T=2 ** 31, gb_rows=2 ** 31) == kda.KDA_ERR_SHAPE
    # a chunk-start state buffer with a negative capacity
    assert _prefill(lib, inter=DUMMY, inter_chunks=-1) == kda.KDA_ERR_SHAPE


def test_decode_host_errors(lib):
    d, g = kda.dims(16), _gate()
    row = 2 * 16 * 128 + 16 * 128

    def call(dims=d, stride=row, pool=DUMMY, idx=DUMMY, B=2):
        return lib.kda_decode_packed(dims, g, DUMMY, stride, DUMMY, DUMMY, B, pool, 240, idx,
                                     DUMMY, None, None)

    assert call(pool=None) == kda.KDA_ERR_NULL_ARG
    assert call(idx=None) == kda.KDA_ERR_NULL_ARG
    assert call(dims=kda.dims(16, K=96)) == kda.KDA_ERR_UNSUPPORTED
    assert call(dims=kda.dims(16, HV=24)) == kda.KDA_ERR_UNSUPPORTED
    assert call(stride=row - 8) == kda.KDA_ERR_SHAPE
    assert call(stride=row + 4) == kda.KDA_ERR_ALIGNMENT
    assert call(B=0) == kda.KDA_OK  # nothing to do, nothing launched


def test_verify_and_commit_host_errors(lib):
    d, g = kda.dims(16), _gate()
    row = 3 * 16 * 128
    assert lib.kda_verify_chain(d, g, DUMMY, row, DUMMY, DUMMY, 2, 0, DUMMY, 240, DUMMY, DUMMY,
                                DUMMY, None, None) == kda.KDA_ERR_SHAPE
    assert lib.kda_verify_chain(d, g, DUMMY, row, DUMMY, DUMMY, 2, 6, DUMMY, 240, DUMMY, DUMMY,
                                None, None, None) == kda.KDA_ERR_NULL_ARG
    assert lib.kda_verify_tree(d, g, DUMMY, row, DUMMY, DUMMY, 2, 6, None, DUMMY, 240, DUMMY,
                               DUMMY, DUMMY, None, None) == kda.KDA_ERR_NULL_ARG
    assert lib.kda_commit(d, DUMMY, 2, 6, DUMMY, None, 240, DUMMY, None, None) == kda.KDA_ERR_NULL_ARG
    assert lib.kda_commit(d, DUMMY, 2, 0, DUMMY, DUMMY, 240, DUMMY, None, None) == kda.KDA_ERR_SHAPE


def test_replay_host_errors(lib):
    d, g = kda.dims(16), _gate()
    row = 3 * 16 * 128
    # ring bytes: [B, T, HV, 388] FP32
    assert lib.kda_replay_ring_bytes(d, 16, 6) == 16 * 6 * 16 * 388 * 4
    assert lib.kda_verify_chain_replay(d, g, DUMMY, row, DUMMY, DUMMY, 2, 0, DUMMY, 240, DUMMY, DUMMY,
                                       DUMMY, None, None) == kda.KDA_ERR_SHAPE
    assert lib.kda_verify_chain_replay(d, g, DUMMY, row, DUMMY, DUMMY, 2, 6, DUMMY, 240, DUMMY, DUMMY,
                                       None, None, None) == kda.KDA_ERR_NULL_ARG
    assert lib.kda_commit_replay(d, None, 2, 6, DUMMY, DUMMY, 240, DUMMY, None, None) == kda.KDA_ERR_NULL_ARG
    assert lib.kda_commit_replay(d, DUMMY, 2, 6, DUMMY, None, 240, DUMMY, None, None) == kda.KDA_ERR_NULL_ARG
    assert lib.kda_commit_replay(d, DUMMY, 2, 0, DUMMY, DUMMY, 240, DUMMY, None, None) == kda.KDA_ERR_SHAPE
    # nothing to do for B = 0
    assert lib.kda_commit_replay(d, None, 0, 6, None, DUMMY, 240, DUMMY, None, None) == kda.KDA_OK


def test_packed_alignment_and_gate_errors(lib):
    """Every 128-bit load of the recurrent kernels needs 16-byte aligned rows,
    pools and rings; the unbounded gate is refused on every path."""
    d, row = kda.dims(16), 3 * 16 * 128
    odd = ctypes.c_void_p(0x10004)

    def decode(gate=None, qkv=DUMMY, a=DUMMY, pool=DUMMY):
        return lib.kda_decode_packed(d, gate or _gate(), qkv, row, a, DUMMY, 2, pool, 240, DUMMY, DUMMY,
                                     None, None)

    assert decode(qkv=odd) == kda.KDA_ERR_ALIGNMENT
    assert decode(a=odd) == kda.KDA_ERR_ALIGNMENT
    assert decode(pool=odd) == kda.KDA_ERR_ALIGNMENT
    assert decode(gate=_gate(A_log=DUMMY, lb=math.nan)) == kda.KDA_ERR_UNSUPPORTED
    assert decode(gate=kda.kda_gate(DUMMY, odd, -5.0, 1, 1, 128 ** -0.5)) == kda.KDA_ERR_ALIGNMENT
    assert lib.kda_verify_chain(d, _gate(), DUMMY, row, DUMMY, DUMMY, 2, 6, odd, 240, DUMMY, DUMMY,
                                DUMMY, None, None) == kda.KDA_ERR_ALIGNMENT
    assert lib.kda_verify_tree(d, _gate(A_log=DUMMY, lb=math.nan), DUMMY, row, DUMMY, DUMMY, 2, 6, DUMMY,
                               DUMMY, 240, DUMMY, DUMMY, DUMMY, None, None) == kda.KDA_ERR_UNSUPPORTED
    assert lib.kda_verify_chain_replay(d, _gate(), DUMMY, row, DUMMY, DUMMY, 2, 6, DUMMY, 240, DUMMY,
                                       DUMMY, odd, None, None) == kda.KDA_ERR_ALIGNMENT
    assert lib.kda_commit_replay(d, odd, 2, 6, DUMMY, DUMMY, 240, DUMMY, None, None) == kda.KDA_ERR_ALIGNMENT
    assert lib.kda_commit_replay(d, DUMMY, 2, 6, DUMMY, odd, 240, DUMMY, None, None) == kda.KDA_ERR_ALIGNMENT
