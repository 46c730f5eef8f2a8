"""Pins of the oracle to facts fixed outside it: the pages' worked example and
rules, closed forms, invariants, exact integer arithmetic, library routines.

Runs on CPU (no ``gpu`` mark). Pages cited: [W] "TokenWeave: Why Hiding
Tensor-Parallel Communication Needs Wave Arithmetic, Not Finer Tiles";
[G] "TokenWeave Guide: Compute-Communication Overlap for LLMs".
"""

import math
import os
import re

import numpy as np
import pytest
import torch

from oracle import bf16, fused, planner, unfused

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                yield line


# --------------------------------------------------------------------------- bf16


def test_bf16_decode_golden_bits():
    for line in _golden_lines("bf16_bits.txt"):
        hx, val = line.split()
        got = bf16.decode(np.array([int(hx, 16)], dtype=np.uint16))[0]
        want = float(val)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), (hx, got, want)


def test_bf16_decode_all_patterns_match_binary32_upper_half():
    # Every finite bf16 pattern, compared with the binary32 value whose upper
    # half it is (the format's definition), decoded by Python's struct module.
    import struct
    pats = [b for b in range(1 << 16) if ((b >> 7) & 0xFF) != 0xFF]
    got = bf16.decode(np.array(pats, dtype=np.uint16))
    want = [struct.unpack("<f", struct.pack("<I", b << 16))[0] for b in pats]
    assert np.array_equal(got, np.array(want, dtype=np.float64))


def test_bf16_rne_golden():
    for line in _golden_lines("bf16_rne.txt"):
        parts = line.split()
        hx = parts[-1]
        expr = " ".join(parts[:-1])
        x = float(eval(expr, {"__builtins__": {}}))  # expressions of powers of two only
        got = int(bf16.encode_rne(np.array([x]))[0])
        assert got == int(hx, 16), (expr, hex(got), hx)


def test_bf16_rne_matches_torch_cast_on_random_fp32():
    # torch's fp32 -> bf16 cast is an independent implementation of the same
    # IEEE rounding; compare on values spanning normal and subnormal ranges.
    rng = np.random.Generator(np.random.PCG64(7))
    raw = rng.integers(0, 1 << 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    x = raw.view(np.float32)
    x = x[np.isfinite(x)]
    ours = bf16.encode_rne(x)
    theirs = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    finite = np.isfinite(bf16.decode(theirs))
    assert np.array_equal(ours[finite], theirs[finite])


def test_bf16_ulp_values():
    assert bf16.ulp(1.0) == 2.0 ** -7
    assert bf16.ulp(1.99) == 2.0 ** -7
    assert bf16.ulp(2.0) == 2.0 ** -6
    assert bf16.ulp(0.75) == 2.0 ** -8
    assert bf16.ulp(-3.0) == 2.0 ** -6
    assert bf16.ulp(1e-40) == 2.0 ** -133
    assert bf16.ulp(0.0) == 2.0 ** -133


# --------------------------------------------------------------------------- RMSNorm


def _z_as_bits(z):
    """Exact bf16 bits of values that are bf16-representable (checked)."""
    b = bf16.encode_rne(np.asarray(z, dtype=np.float64))
    assert np.array_equal(bf16.decode(b), np.asarray(z, dtype=np.float64))
    return b


def _parse_kv(tokens):
    out = {}
    for t in tokens:
        k, v = t.split("=", 1)
        out[k] = v
    return out


def _gamma(spec, h):
    if spec.startswith("all:"):
        return [float(spec[4:])] * h
    g = [float(v) for v in spec.split(",")]
    assert len(g) == h
    return g


def test_rmsnorm_closed_forms():
    """Closed forms through the full fused oracle with N=1, R=0 (so z = P_0)."""
    seen = set()
    for line in _golden_lines("rmsnorm_closed_forms.txt"):
        kind, *rest = line.split()
        kv = _parse_kv(rest)
        eps = float(kv["eps"])
        if kind == "h2_34":
            z = [float(v) for v in kv["z"].split(",")]
            g = [float(v) for v in kv["gamma"].split(",")]
            want = [float(v) for v in kv["y"].split(",")]
            want_exact = [3 / math.sqrt(12.5), 4 / math.sqrt(12.5)]
            assert np.allclose(want, want_exact, rtol=0, atol=1e-15)
        elif kind == "const":
            c, h = float(kv["c"]), int(kv["H"])
            z = [c] * h
            g = _gamma(kv["gamma"], h)
            want = [gi * c / math.sqrt(c * c + eps) for gi in g]
        elif kind == "onehot":
            c, h, k = float(kv["c"]), int(kv["H"]), int(kv["k"])
            z = [0.0] * h
            z[k] = c
            g = _gamma(kv["gamma"], h)
            want = [0.0] * h
            want[k] = g[k] * c / math.sqrt(c * c / h + eps)
        elif kind == "zero":
            h = int(kv["H"])
            z = [0.0] * h
            g = _gamma(kv["gamma"], h)
            want = [0.0] * h
        else:
            raise AssertionError(kind)
        seen.add(kind)
        pb = _z_as_bits(z)[None, None, :]          # N=1, T=1
        rb = _z_as_bits([0.0] * len(z))[None, :]
        gb = _z_as_bits(g)
        z64, y64 = fused.reduce_residual_rmsnorm(pb, rb, gb, eps)
        assert np.array_equal(z64[0], np.array(z))
        assert np.allclose(y64[0], want, rtol=1e-14, atol=0), (kind, y64[0], want)
        assert not np.isnan(y64).any()
    assert seen == {"h2_34", "const", "onehot", "zero"}


def test_rmsnorm_mean_square_invariant():
    """mean_j (y_j / gamma_j)^2 = ms / (ms + eps), ms = mean(z^2): a property of
    the formula of [G] "The Standard RMSNorm Memory Round-Trip"."""
    rng = np.random.Generator(np.random.PCG64(3))
    for h, eps in [(64, 1e-5), (4096, 1e-5), (8, 0.5)]:
        z = rng.standard_normal((5, h)) * rng.uniform(0.01, 10, size=(5, 1))
        g = rng.uniform(0.5, 1.5, size=h)
        y = fused.rms_norm(z, g, eps)
        ms = np.mean(z * z, axis=1)
        lhs = np.mean((y / g) ** 2, axis=1)
        assert np.allclose(lhs, ms / (ms + eps), rtol=1e-12)


def test_rmsnorm_scale_invariance_at_eps_zero():
    """With eps = 0 RMSNorm is invariant to scaling its input by any c > 0."""
    rng = np.random.Generator(np.random.PCG64(4))
    z = rng.standard_normal((3, 32))
    g = rng.uniform(0.5, 1.5, size=32)
    assert np.allclose(fused.rms_norm(z, g, 0.0), fused.rms_norm(37.5 * z, g, 0.0), rtol=1e-13)
    assert np.allclose(fused.rms_norm(z, g, 0.0), -fused.rms_norm(-z, g, 0.0), rtol=0, atol=0)


def test_rmsnorm_gamma_enters_per_element():
    """Swapping two hidden positions of z and gamma swaps the same outputs."""
    rng = np.random.Generator(np.random.PCG64(5))
    z = rng.standard_normal((2, 16))
    g = rng.uniform(0.5, 1.5, size=16)
    y = fused.rms_norm(z, g, 1e-5)
    perm = np.arange(16)
    perm[[2, 11]] = perm[[11, 2]]
    y2 = fused.rms_norm(z[:, perm], g[perm], 1e-5)
    assert np.array_equal(y[:, perm], y2)


# --------------------------------------------------------------------------- reduce + residual


def test_reduce_small_integers_exact():
    """Partials and residual drawn from small integers: every sum is exact in
    bf16, fp32 and fp64, so z and the updated residual equal Python's integer
    sums (ranks summed then the residual added, [W] "Fix two")."""
    rng = np.random.Generator(np.random.PCG64(11))
    n, t, h = 8, 5, 24
    pi = rng.integers(-4, 5, size=(n, t, h))
    ri = rng.integers(-4, 5, size=(t, h))
    pb = _z_as_bits(pi.astype(np.float64).ravel()).reshape(n, t, h)
    rb = _z_as_bits(ri.astype(np.float64).ravel()).reshape(t, h)
    gb = _z_as_bits(np.ones(h))
    z64, y64 = fused.reduce_residual_rmsnorm(pb, rb, gb, 1e-5)
    want = [[sum(int(pi[r, a, b]) for r in range(n)) + int(ri[a, b]) for b in range(h)] for a in range(t)]
    assert np.array_equal(z64, np.array(want, dtype=np.float64))
    res = fused.residual_fp32_rank_order(pb, rb)
    assert np.array_equal(bf16.decode(res), np.array(want, dtype=np.float64))
    # each normalised row by the formula, written out with Python floats
    for a in range(t):
        ms = sum(v * v for v in want[a]) / h
        for b in range(h):
            assert math.isclose(y64[a, b], want[a][b] / math.sqrt(ms + 1e-5), rel_tol=1e-14, abs_tol=1e-300)


def test_residual_fp32_rank_order_is_left_to_right():
    """A case built by hand whose bf16 result depends on the summation order.

    P_0 = 1, P_1 = P_2 = 2^-24, P_3 = 2^-8, R = 0.  In fp32, 1 + 2^-24 is a tie
    and rounds to even (1), twice; then 1 + 2^-8 is exact; bf16(1 + 2^-8) is a
    tie and rounds to even: 0x3F80.  The exact sum 1 + 2^-8 + 2^-23 rounds up
    to 0x3F81, and so would the reversed order.
    """
    vals = [1.0, 2.0 ** -24, 2.0 ** -24, 2.0 ** -8]
    pb = _z_as_bits(vals).reshape(4, 1, 1)
    rb = _z_as_bits([0.0]).reshape(1, 1)
    assert int(fused.residual_fp32_rank_order(pb, rb)[0, 0]) == 0x3F80
    z64 = fused.reduce_residual(pb, rb)
    assert z64[0, 0] == 1 + 2.0 ** -8 + 2.0 ** -23
    assert int(bf16.encode_rne(z64)[0, 0]) == 0x3F81
    # residual added last: with P = (1, 2^-24) and R = 2^-24 the fp32 result is 1 (tie twice)
    pb2 = _z_as_bits([1.0, 2.0 ** -24]).reshape(2, 1, 1)
    rb2 = _z_as_bits([2.0 ** -24]).reshape(1, 1)
    assert int(fused.residual_fp32_rank_order(pb2, rb2)[0, 0]) == 0x3F80


def test_residual_within_one_ulp_of_exact_on_workload_like_data():
    rng = np.random.Generator(np.random.PCG64(12))
    n, t, h = 8, 16, 256
    pb = bf16.encode_rne(rng.standard_normal((n, t, h)) * 0.02)
    rb = bf16.encode_rne(rng.standard_normal((t, h)))
    z64 = fused.reduce_residual(pb, rb)
    r32 = bf16.decode(fused.residual_fp32_rank_order(pb, rb))
    assert np.all(np.abs(r32 - z64) <= bf16.ulp(z64))


def test_shard_invariance_oracle():
    """Normalising token-contiguous shards equals normalising the whole batch
    ([W] "Fix two": per-token norm after a token-boundary reduce-scatter)."""
    rng = np.random.Generator(np.random.PCG64(13))
    t, h = 96, 64
    z = rng.standard_normal((t, h))
    gb = bf16.encode_rne(rng.uniform(0.5, 1.5, size=h))
    whole = fused.rms_norm(z, bf16.decode(gb), 1e-5)
    for shard in (1, 8, 12, 32, 50, 96, 200):
        assert np.array_equal(fused.normalize_shards(z, gb, 1e-5, shard), whole)


def test_unfused_oracle_small_integers():
    rng = np.random.Generator(np.random.PCG64(14))
    n, t, h = 4, 3, 16
    pi = rng.integers(-4, 5, size=(n, t, h)).astype(np.float64)
    ri = rng.integers(-4, 5, size=(t, h)).astype(np.float64)
    pb = bf16.encode_rne(pi)
    rb = bf16.encode_rne(ri)
    s, rnew, y = unfused.reduce_then_rmsnorm(pb, rb, bf16.encode_rne(np.ones(h)), 1e-5)
    assert np.array_equal(bf16.decode(s), pi.sum(axis=0))
    assert np.array_equal(bf16.decode(rnew), pi.sum(axis=0) + ri)
    z = pi.sum(axis=0) + ri
    for a in range(t):
        ms = float(np.sum(z[a] ** 2)) / h
        assert np.allclose(y[a], z[a] / math.sqrt(ms + 1e-5), rtol=1e-14, atol=0)


def test_unfused_intermediate_rounds_the_partial_sum():
    """The unfused path rounds the partial sum to bf16 before adding the
    residual (its HBM round trip): 1 + 2^-8 (a bf16 tie -> 1) plus R = 2^-8
    gives 1 + 2^-8 -> bf16 1.0, while the fused path keeps the fp32 sum
    1 + 2^-7 exactly."""
    pb = bf16.encode_rne(np.array([1.0, 2.0 ** -8])).reshape(2, 1, 1)
    rb = bf16.encode_rne(np.array([2.0 ** -8])).reshape(1, 1)
    s, rnew, _ = unfused.reduce_then_rmsnorm(pb, rb, bf16.encode_rne(np.ones(1)), 1e-5)
    assert int(s[0, 0]) == 0x3F80
    assert int(rnew[0, 0]) == 0x3F80
    assert int(fused.residual_fp32_rank_order(pb, rb)[0, 0]) == 0x3F81


# --------------------------------------------------------------------------- planner


def _planner_cases():
    for line in _golden_lines("planner_pins.txt"):
        lhs, rhs = line.split("->")
        T, C, S, offs, mins = lhs.split()
        p, s = rhs.split()
        offsets = None if offs == "all" else planner.DEFAULT_OFFSETS
        assert offs in ("all", "default")
        yield int(T), int(C), int(S), offsets, int(mins), int(p), int(s)


def test_planner_golden():
    n = 0
    for T, C, S, offsets, mins, p, s in _planner_cases():
        assert planner.wave_split(T, C, S, offsets, mins) == (p, s), (T, C, S)
        n += 1
    assert n >= 15


def test_planner_worked_example_wave_counts():
    """[W] "The overlap trap": 300 CTAs on 132 SMs: unsplit 132+132+36 = 3 waves;
    150/150 = 2 + 2 = 4 waves; "Fix one": 132/168 = 1 + 2 = 3 waves."""
    assert planner.waves(300, 132) == 3
    assert planner.waves(150, 132) + planner.waves(150, 132) == 4
    assert planner.waves(132, 132) + planner.waves(168, 132) == 3
    assert not planner.feasible(150, 300, 300, 132)
    assert planner.feasible(132, 300, 300, 132)
    # the default offset grid cannot reach 132/168 (needs offset 18); its first
    # admissible candidate is offset 64: 86 (1 wave) / 214 (2 waves)
    assert planner.wave_split(300, 300, 132, planner.DEFAULT_OFFSETS, 0) == (86, 214)


def test_planner_split_conserves_tokens_and_waves():
    rng = np.random.Generator(np.random.PCG64(21))
    for _ in range(300):
        T = int(rng.integers(0, 3000))
        C = int(rng.integers(0, 400))
        S = int(rng.integers(1, 200))
        p, s = planner.wave_split(T, C, S)
        assert p + s == T and p >= 0 and s >= 0
        if s:
            assert planner.feasible(p, T, C, S)
            assert abs(p - T // 2) in planner.DEFAULT_OFFSETS and T >= 1024


def test_planner_rejects_bad_args():
    with pytest.raises(ValueError):
        planner.wave_split(10, 5, 0)
    with pytest.raises(ValueError):
        planner.wave_split(10, -1, 4)
    with pytest.raises(ValueError):
        planner.wave_split(-1, 5, 4)
    with pytest.raises(ValueError):
        planner.wave_split(2048, 500, 100, offsets=(0, -64))


def test_golden_files_cite_sources():
    for name in ("planner_pins.txt", "bf16_bits.txt", "bf16_rne.txt", "rmsnorm_closed_forms.txt"):
        text = open(os.path.join(GOLDEN, name)).read()
        assert re.search(r"\[(W|G)\]|IEEE", text), name


def test_fp64_oracle_against_50_digit_decimal_reference():
    """The fp64 oracle against exact decimal arithmetic (50 digits): the sum of
    bf16 values is exact in Decimal, the mean square and square root are
    correctly rounded at 50 digits. Rows include heavy cancellation and
    outliers. The oracle must agree to 1e-12 relative (it is the reference the
    GPU is held to within 2 bf16 ulps, ~8e-3)."""
    from decimal import Decimal, getcontext
    getcontext().prec = 50
    rng = np.random.Generator(np.random.PCG64(50))
    n, t, h = 4, 6, 96
    p = rng.standard_normal((n, t, h)) * 0.02
    p[:, 2] *= 1e4                       # large partials ...
    p[3, 2] = -p[:3, 2].sum(axis=0)      # ... that nearly cancel
    r = rng.standard_normal((t, h))
    r[4, ::7] *= 300.0                   # outliers
    pb, rb = bf16.encode_rne(p), bf16.encode_rne(r)
    gb = bf16.encode_rne(rng.uniform(0.5, 1.5, size=h))
    eps = 1e-5
    z64, y64 = fused.reduce_residual_rmsnorm(pb, rb, gb, eps)
    P, R, G = bf16.decode(pb), bf16.decode(rb), bf16.decode(gb)
    for a in range(t):
        z = [sum((Decimal(float(P[k, a, b])) for k in range(n)), Decimal(float(R[a, b])))
             for b in range(h)]
        ms = sum(v * v for v in z) / h
        scale = (ms + Decimal(eps)).sqrt()
        for b in range(h):
            y = z[b] / scale * Decimal(float(G[b]))
            assert float(z[b]) == z64[a, b]
            if y != 0:
                assert abs(float(y) - y64[a, b]) <= 1e-12 * abs(float(y)), (a, b)
            else:
                assert y64[a, b] == 0


# ------------------------------------------------------------------ token-boundary shards

def test_shard_oracle_hand_cases():
    """Hand-computed shards: the Llama-3.3-70B configuration's 8 x 128-token
    shards, an uneven batch whose last rank owns nothing, and a single rank."""
    from oracle import shards
    assert [shards.shard_rows(1024, 8, r) for r in range(8)] == [(128 * r, 128) for r in range(8)]
    assert [shards.shard_rows(5, 4, r) for r in range(4)] == [(0, 2), (2, 2), (4, 1), (5, 0)]
    assert [shards.shard_rows(10, 3, r) for r in range(3)] == [(0, 4), (4, 4), (8, 2)]
    assert shards.shard_rows(7, 1, 0) == (0, 7)
    assert shards.shard_rows(0, 4, 2) == (0, 0)


def test_shard_oracle_partition_invariants():
    """For every T <= 70 and world <= 9: the shards are contiguous, in rank
    order, cover every row exactly once, and hold ceil(T / world) rows each
    except the tail. A mistake in the owner rule (floor for ceil, an offset
    by one rank, interleaved rows) breaks one of these."""
    from oracle import shards
    for T in range(0, 71):
        for world in range(1, 10):
            s = -(-T // world)
            got = [shards.shard_rows(T, world, r) for r in range(world)]
            covered = []
            nxt = 0
            for r, (row0, rows) in enumerate(got):
                assert rows >= 0 and row0 == min(nxt, T)
                covered.extend(range(row0, row0 + rows))
                nxt = row0 + rows
                assert rows <= s
                if nxt < T:
                    assert rows == s
            assert covered == list(range(T))
