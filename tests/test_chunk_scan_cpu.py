"""Chunk-parallel state passing, checked in FP64 and FP32 on the CPU.

The prefill's state pass is a chain over a sequence's chunks.  Each chunk's
end state is affine in its start state, S_end = M_c S_start + B_c (the maps
are written out in tests/chunk_form.py, from the chunk form of the gated delta
rule), so the chunk-start states are prefix compositions of the maps and a
scan finds them in log2(chunks) levels.  These tests pin the facts a parallel
pass would rely on:
  * the scan gives the sequential chunk form's states, to FP64 rounding;
  * ||M_c||_2 <= exp(sum over the chunk's tokens of max_c g_t[c]), since every
    token's factor (I - beta k k^T) Diag(e^g) has norm <= max e^g when
    ||k|| = 1 and 0 <= beta <= 1; so a window of h chunks started from zero
    misses the true state by at most the product of h such bounds times the
    state at the window's start;
  * the scan run in FP32 stays far inside the state tolerance (1e-3 x RMS);
  * on tensor cores its products need split operands: TF32 alone misses the
    tolerance when the decay is slow, three TF32 products (hi/lo) do not;
  * the grouped three-stage pass (tests/chunk_form.py, grouped_prefill), which
    needs no per-chunk storage, gives the sequential outputs and states.
"""
import numpy as np

from tests.chunk_form import chunk_maps, chunk_prefill, grouped_prefill, scan_chunk_states


def _inputs(T, K, lower_bound, seed):
    """Folded inputs: unit q and k, the bounded gate g = lb * sigmoid(e^{A_log}
    (a + dt_bias)) with a ~ N(0, 1), beta = sigmoid(N(0, 1))."""
    rng = np.random.default_rng(seed)
    sig = lambda x: 1.0 / (1.0 + np.exp(-x))
    unit = lambda x: x / np.linalg.norm(x, axis=1, keepdims=True)
    q, k = unit(rng.standard_normal((T, K))), unit(rng.standard_normal((T, K)))
    v = rng.standard_normal((T, K))
    A_log, dt_bias = rng.uniform(-1, 1), rng.normal(0, 0.1, K)
    g = lower_bound * sig(np.exp(A_log) * (rng.standard_normal((T, K)) + dt_bias))
    beta = sig(rng.standard_normal(T))
    S0 = rng.normal(0, 0.02, (K, K))
    return q, k, v, g, beta, S0


def test_scan_equals_sequential_chunk_form():
    # 14 chunks (not a power of two), ragged last chunk, slow decay so that
    # every map matters
    q, k, v, g, beta, S0 = _inputs(64 * 13 + 5, 32, -0.05, seed=1)
    _, S_T, starts = chunk_prefill(q, k, v, g, beta, S0, 32 ** -0.5)
    maps = chunk_maps(q, k, v, g, beta)
    assert max(np.linalg.norm(m, 2) for m, _ in maps) > 0.1
    scan_starts, scan_T = scan_chunk_states(maps, S0)
    rms = np.sqrt(np.mean(np.square(starts)))
    assert len(scan_starts) == len(starts) == 14
    np.testing.assert_allclose(np.array(scan_starts), np.array(starts), rtol=0, atol=1e-12 * rms)
    np.testing.assert_allclose(scan_T, S_T, rtol=0, atol=1e-12 * rms)


def _norm_bounds(g, chunk=64):
    return [float(np.exp(np.sum(np.max(g[s:s + chunk], axis=1)))) for s in range(0, g.shape[0], chunk)]


def test_map_norm_bound_and_truncated_windows():
    for lb in (-5.0, -0.05):
        q, k, v, g, beta, S0 = _inputs(64 * 10, 32, lb, seed=2)
        _, _, starts = chunk_prefill(q, k, v, g, beta, S0, 32 ** -0.5)
        maps = chunk_maps(q, k, v, g, beta)
        bounds = _norm_bounds(g)
        for (m, _), bound in zip(maps, bounds):
            assert np.linalg.norm(m, 2) <= bound * (1 + 1e-12)
        # the start state of chunk c from only the h chunks before it, begun
        # from zero, against the true one
        for h in (1, 2, 3):
            for c in range(h, len(maps)):
                S = np.zeros_like(S0)
                for j in range(c - h, c):
                    S = maps[j][0] @ S + maps[j][1]
                err = np.linalg.norm(S - starts[c])
                assert err <= np.prod(bounds[c - h:c]) * np.linalg.norm(starts[c - h]) * (1 + 1e-9) + 1e-13


def test_strong_gate_makes_one_chunk_enough():
    """At the benchmarks' gate (lower bound -5) a chunk's end state does not
    depend on its start state at FP32 precision: every map is below 1e-30."""
    q, k, v, g, beta, _ = _inputs(64 * 8, 128, -5.0, seed=3)
    assert max(np.linalg.norm(m, 2) for m, _ in chunk_maps(q, k, v, g, beta)) < 1e-30


def test_fp32_scan_within_state_tolerance():
    # the slowest decay tried: the maps stay close to 1 in norm
    q, k, v, g, beta, S0 = _inputs(64 * 16, 128, -0.005, seed=4)
    _, _, starts = chunk_prefill(q, k, v, g, beta, S0, 128 ** -0.5)
    maps = chunk_maps(q, k, v, g, beta)
    assert max(np.linalg.norm(m, 2) for m, _ in maps) > 0.5
    st32, _ = scan_chunk_states([(m.astype(np.float32), b.astype(np.float32)) for m, b in maps], S0)
    ref = np.array(starts)
    rms = np.sqrt(np.mean(np.square(ref)))
    assert np.max(np.abs(np.array(st32, np.float64) - ref)) <= 1e-5 * rms


def _tf32(x):
    """FP32 rounded to TF32 (10 mantissa bits), to nearest even."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0xFFF + ((u >> 13) & 1)) & ~np.uint64(0x1FFF)
    return u.astype(np.uint32).view(np.float32)


def _scan_with(maps, S0, mm):
    """scan_chunk_states with every product done by mm (FP32 results)."""
    Mp, Bp = [m for m, _ in maps], [b for _, b in maps]
    n, d = len(maps), 1
    while d < n:
        Mn, Bn = list(Mp), list(Bp)
        for c in range(d, n):
            Mn[c] = mm(Mp[c], Mp[c - d])
            Bn[c] = (mm(Mp[c], Bp[c - d]).astype(np.float64) + Bp[c]).astype(np.float32)
        Mp, Bp, d = Mn, Bn, 2 * d
    S0 = np.asarray(S0, np.float32)
    return [S0] + [(mm(Mp[c], S0).astype(np.float64) + Bp[c]).astype(np.float32) for c in range(n - 1)]


def test_tensor_core_scan_needs_split_operands():
    """The scan's products on tensor cores: with TF32 operands (FP32
    accumulation) the chunk-start states miss the state tolerance when the
    decay is slow; with each operand split into TF32 hi + lo and three
    products (dropping lo x lo) they stay far inside it."""
    f64 = lambda x: x.astype(np.float64)

    def tf32_mm(a, b):
        return (f64(_tf32(a)) @ f64(_tf32(b))).astype(np.float32)

    def split_mm(a, b):
        ah, bh = _tf32(a), _tf32(b)
        al, bl = _tf32(np.float32(a) - ah), _tf32(np.float32(b) - bh)
        return (f64(ah) @ f64(bh) + f64(ah) @ f64(bl) + f64(al) @ f64(bh)).astype(np.float32)

    q, k, v, g, beta, S0 = _inputs(4096, 128, -0.005, seed=4)
    _, _, starts = chunk_prefill(q, k, v, g, beta, S0, 128 ** -0.5)
    maps = [(m.astype(np.float32), b.astype(np.float32)) for m, b in chunk_maps(q, k, v, g, beta)]
    ref = np.array(starts)
    rms = np.sqrt(np.mean(np.square(ref)))
    err = lambda st: np.max(np.abs(np.array(st, np.float64) - ref)) / rms
    assert err(_scan_with(maps, S0, tf32_mm)) > 1e-3
    assert err(_scan_with(maps, S0, split_mm)) < 1e-5


def test_grouped_pass_equals_sequential_chunk_form():
    """The three-stage grouped pass (groups from zero with the identity
    carried, a short chain over group starts, groups rerun from their true
    starts) gives the sequential chunk form's outputs and states, for group
    sizes that divide the chunk count and ones that do not."""
    q, k, v, g, beta, S0 = _inputs(64 * 11 + 9, 32, -0.05, seed=5)
    o, S_T, starts = chunk_prefill(q, k, v, g, beta, S0, 32 ** -0.5)
    orms, srms = np.sqrt(np.mean(np.square(o))), np.sqrt(np.mean(np.square(starts)))
    for group in (1, 3, 4, 12, 20):
        og, Sg, stg = grouped_prefill(q, k, v, g, beta, S0, 32 ** -0.5, group=group)
        np.testing.assert_allclose(og, o, rtol=0, atol=1e-12 * orms)
        np.testing.assert_allclose(np.array(stg), np.array(starts), rtol=0, atol=1e-12 * srms)
        np.testing.assert_allclose(Sg, S_T, rtol=0, atol=1e-12 * srms)
