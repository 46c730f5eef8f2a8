"""Plant plausible mistakes in the oracle (on the CPU, by monkeypatching) and
check that at least one pin in test_oracle_pins.py fails for each. This shows
the pins constrain every term of the oracle, not only that they pass."""

import numpy as np
import pytest

from oracle import bf16, fused, planner

import test_oracle_pins as pins


def _fails(*checks):
    for check in checks:
        try:
            check()
        except AssertionError:
            return True
    return False


NORM_PINS = (pins.test_rmsnorm_closed_forms, pins.test_reduce_small_integers_exact,
             pins.test_rmsnorm_mean_square_invariant)


def _rms_eps_outside(z, gamma, eps):
    z = np.asarray(z, dtype=np.float64)
    ms = np.sum(z * z, axis=-1, keepdims=True) / z.shape[-1]
    return z / (np.sqrt(ms) + eps) * np.asarray(gamma, dtype=np.float64)


def _rms_divisor_h_minus_1(z, gamma, eps):
    z = np.asarray(z, dtype=np.float64)
    ms = np.sum(z * z, axis=-1, keepdims=True) / max(z.shape[-1] - 1, 1)
    return z / np.sqrt(ms + eps) * np.asarray(gamma, dtype=np.float64)


def _rms_no_gamma(z, gamma, eps):
    z = np.asarray(z, dtype=np.float64)
    ms = np.sum(z * z, axis=-1, keepdims=True) / z.shape[-1]
    return z / np.sqrt(ms + eps)


def _rms_no_sqrt(z, gamma, eps):
    z = np.asarray(z, dtype=np.float64)
    ms = np.sum(z * z, axis=-1, keepdims=True) / z.shape[-1]
    return z / (ms + eps) * np.asarray(gamma, dtype=np.float64)


def _rms_gamma_reversed(z, gamma, eps):
    z = np.asarray(z, dtype=np.float64)
    ms = np.sum(z * z, axis=-1, keepdims=True) / z.shape[-1]
    return z / np.sqrt(ms + eps) * np.asarray(gamma, dtype=np.float64)[::-1]


@pytest.mark.parametrize("mutant", [_rms_eps_outside, _rms_divisor_h_minus_1, _rms_no_gamma,
                                    _rms_no_sqrt, _rms_gamma_reversed])
def test_norm_mutants_are_caught(monkeypatch, mutant):
    monkeypatch.setattr(fused, "rms_norm", mutant)
    assert _fails(*NORM_PINS)


def _reduce_drops_residual(partials, residual):
    p = np.asarray(partials)
    p = p[None] if p.ndim == 2 else p
    z = np.zeros(np.asarray(residual).shape)
    for r in range(p.shape[0]):
        z = z + bf16.decode(p[r])
    return z


def _reduce_drops_last_rank(partials, residual):
    p = np.asarray(partials)
    p = p[None] if p.ndim == 2 else p
    z = bf16.decode(residual)
    for r in range(p.shape[0] - 1):
        z = z + bf16.decode(p[r])
    return z


def _reduce_subtracts_residual(partials, residual):
    p = np.asarray(partials)
    p = p[None] if p.ndim == 2 else p
    z = -bf16.decode(residual)
    for r in range(p.shape[0]):
        z = z + bf16.decode(p[r])
    return z


@pytest.mark.parametrize("mutant", [_reduce_drops_residual, _reduce_drops_last_rank,
                                    _reduce_subtracts_residual])
def test_reduce_mutants_are_caught(monkeypatch, mutant):
    monkeypatch.setattr(fused, "reduce_residual", mutant)
    assert _fails(pins.test_reduce_small_integers_exact)


def _res_reverse_order(partials, residual):
    p = np.asarray(partials)
    p = p[None] if p.ndim == 2 else p
    acc = bf16.decode(residual).astype(np.float32)
    for r in range(p.shape[0] - 1, -1, -1):
        acc = (acc + bf16.decode(p[r]).astype(np.float32)).astype(np.float32)
    return bf16.encode_rne(acc)


def _res_in_fp64(partials, residual):
    return bf16.encode_rne(fused.reduce_residual(partials, residual))


@pytest.mark.parametrize("mutant", [_res_reverse_order, _res_in_fp64])
def test_residual_order_mutants_are_caught(monkeypatch, mutant):
    monkeypatch.setattr(fused, "residual_fp32_rank_order", mutant)
    assert _fails(pins.test_residual_fp32_rank_order_is_left_to_right)


def _encode_truncate(x):
    v = np.asarray(x, dtype=np.float64).astype(np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)


def _encode_ties_away(x):
    x = np.asarray(x, dtype=np.float64)
    u = bf16.ulp(x)
    q = x / u
    v = (np.sign(q) * np.floor(np.abs(q) + 0.5)) * u
    v = np.where(np.abs(v) > bf16.BF16_MAX, np.copysign(np.inf, x), v)
    return (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("mutant", [_encode_truncate, _encode_ties_away])
def test_bf16_rounding_mutants_are_caught(monkeypatch, mutant):
    monkeypatch.setattr(bf16, "encode_rne", mutant)
    assert _fails(pins.test_bf16_rne_golden)


def _waves_floor(c, S):
    return c // S


def _ctas_floor(t, T, C):
    return (t * C) // T if T else 0


@pytest.mark.parametrize("name,mutant", [("waves", _waves_floor), ("ctas", _ctas_floor)])
def test_planner_arithmetic_mutants_are_caught(monkeypatch, name, mutant):
    monkeypatch.setattr(planner, name, mutant)
    assert _fails(pins.test_planner_golden, pins.test_planner_worked_example_wave_counts)


def test_planner_tie_break_mutant_is_caught(monkeypatch):
    orig = planner.wave_split

    def larger_prefix_first(T, C, S, offsets=planner.DEFAULT_OFFSETS,
                            min_split_tokens=planner.DEFAULT_MIN_SPLIT_TOKENS):
        p, s = orig(T, C, S, offsets, min_split_tokens)
        return (s, p) if s else (p, s)  # mirror: the larger piece first

    monkeypatch.setattr(planner, "wave_split", larger_prefix_first)
    assert _fails(pins.test_planner_golden)


def test_planner_threshold_mutant_is_caught(monkeypatch):
    orig = planner.wave_split

    def no_threshold(T, C, S, offsets=planner.DEFAULT_OFFSETS, min_split_tokens=0):
        return orig(T, C, S, offsets, 0)

    monkeypatch.setattr(planner, "wave_split", no_threshold)
    assert _fails(pins.test_planner_golden)


SHARD_PINS = (pins.test_shard_oracle_hand_cases, pins.test_shard_oracle_partition_invariants)


def _owner_floor(t, T, world):
    return t // max(T // world, 1)          # floor for ceil


def _owner_interleaved(t, T, world):
    return t % world                         # round-robin rows, not token ranges


def _owner_reversed(t, T, world):
    return world - 1 - t // -(-T // world)   # shards in reverse rank order


@pytest.mark.parametrize("mutant", [_owner_floor, _owner_interleaved, _owner_reversed])
def test_shard_mutants_are_caught(monkeypatch, mutant):
    from oracle import shards
    monkeypatch.setattr(shards, "owner", mutant)
    assert _fails(*SHARD_PINS)
