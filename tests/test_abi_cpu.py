"""The C-ABI library on the CPU: it loads, exports every symbol the header
declares, its host-only planner equals the brute-force oracle, and argument
validation returns status codes before any CUDA call (no GPU is touched:
pointers here are fake addresses that validation never dereferences)."""

import ctypes
import math
import os
import re

import numpy as np
import pytest

import reduce_rmsnorm_gb300 as tw
from oracle import planner as oplanner

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from reduce_rmsnorm_gb300 import build
    build.build()
    return tw.lib()


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "tw.h")).read()
    return sorted(set(re.findall(r"^TW_API\s+(?:int|const char\*)\s+(tw_\w+)\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    syms = _declared_symbols()
    for name in ("tw_fused_reduce_residual_rmsnorm", "tw_wave_split", "tw_run_split", "tw_strerror"):
        assert name in syms


def test_library_exports_every_declared_symbol(L):
    for name in _declared_symbols():
        assert hasattr(L, name), name
    assert set(_declared_symbols()) <= set(tw.EXPORTED) | set()
    for name in tw.EXPORTED:
        assert name in _declared_symbols(), name


def test_library_exports_only_the_declared_entry_points(L):
    import shutil
    import subprocess
    if shutil.which("nm") is None:
        pytest.skip("needs nm")
    out = subprocess.run(["nm", "-D", "--defined-only", tw.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    names = {line.split()[-1] for line in out.splitlines() if line.strip()}
    assert names == set(_declared_symbols()), sorted(names ^ set(_declared_symbols()))


def test_strerror(L):
    for code in range(6):
        assert tw.tw_strerror(code).startswith("TW_")
    assert "unknown" in tw.tw_strerror(99)


# ------------------------------------------------------------------ planner (pure host)


def _golden_planner_cases():
    path = os.path.join(ROOT, "tests", "golden", "planner_pins.txt")
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        lhs, rhs = line.split("->")
        T, C, S, offs, mins = lhs.split()
        p, s = rhs.split()
        yield int(T), int(C), int(S), (None if offs == "all" else tw.DEFAULT_OFFSETS), int(mins), int(p), int(s)


def test_planner_golden(L):
    for T, C, S, offs, mins, p, s in _golden_planner_cases():
        assert tw.tw_wave_split(T, C, S, offs, mins) == (p, s), (T, C, S)


def test_planner_configs_at_148_sms(L):
    # Token counts of the split workload; C = ceil(T/128) * (8192/128) / 8.
    for T, want in [(1024, (1024, 0)), (2048, (2048, 0)), (4096, (2048, 2048)), (8192, (4096, 4096))]:
        C = math.ceil(T / 128) * (8192 // 128) // 8
        assert tw.tw_wave_split(T, C, 148) == want
        assert oplanner.wave_split(T, C, 148) == want


def test_planner_exhaustive_small_every_offset(L):
    """Every (T, C, S) with T <= 40, C <= 40, S <= 20, every integer offset, no threshold."""
    n = 0
    for T in range(0, 41):
        for C in range(0, 41):
            for S in range(1, 21):
                want = oplanner.wave_split(T, C, S, None, 0)
                assert tw.tw_wave_split(T, C, S, None, 0) == want, (T, C, S)
                n += 1
    assert n == 41 * 41 * 20


def test_planner_random_default_grid(L):
    rng = np.random.Generator(np.random.PCG64(2024))
    for _ in range(600):
        T = int(rng.integers(0, 6000))
        C = int(rng.integers(0, 1200))
        S = int(rng.integers(1, 300))
        mins = int(rng.choice([0, 512, 1024, 4096]))
        assert tw.tw_wave_split(T, C, S, tw.DEFAULT_OFFSETS, mins) == \
            oplanner.wave_split(T, C, S, tw.DEFAULT_OFFSETS, mins), (T, C, S, mins)


def test_planner_on_the_projection_cta_formula(L):
    """The C planner equals the brute-force oracle on the CTA counts of the
    row-parallel projection, C = ceil(T/128) * (H/128) / 8: every token count
    1024..9600 at H = 8192 on 148 SMs, and for H = 4096, 8192, 16384 on 132,
    144, 148 and 152 SMs every count 1024..2048 plus a stride-37 sweep to
    9600. The plans taken must use every offset of the default grid."""
    cases = [(T, 8192, 148) for T in range(1024, 9601)]
    cases += [(T, H, S) for H in (4096, 8192, 16384) for S in (132, 144, 148, 152)
              for T in list(range(1024, 2049)) + list(range(2049, 9601, 37))]
    used = set()
    for T, H, S in cases:
        C = math.ceil(T / 128) * (H // 128) // 8
        want = oplanner.wave_split(T, C, S)
        assert tw.tw_wave_split(T, C, S) == want, (T, H, S)
        if want[1] > 0:
            used.add(abs(want[0] - T // 2))
    assert used == set(tw.DEFAULT_OFFSETS), sorted(used)


def test_planner_custom_offsets_unsorted_duplicates(L):
    rng = np.random.Generator(np.random.PCG64(99))
    for _ in range(200):
        offs = [int(x) for x in rng.integers(0, 700, size=int(rng.integers(1, 8)))]
        offs += offs[:2]
        T = int(rng.integers(1024, 5000))
        C = int(rng.integers(1, 900))
        S = int(rng.integers(1, 200))
        assert tw.tw_wave_split(T, C, S, offs, 1024) == oplanner.wave_split(T, C, S, offs, 1024)


def test_planner_rejects_bad_args(L):
    bad = [(-1, 5, 4, tw.DEFAULT_OFFSETS), (10, -1, 4, tw.DEFAULT_OFFSETS),
           (10, 5, 0, tw.DEFAULT_OFFSETS), (2048, 500, 100, (0, -64))]
    for T, C, S, offs in bad:
        with pytest.raises(tw.TwError) as e:
            tw.tw_wave_split(T, C, S, offs)
        assert e.value.status == tw.TW_ERR_INVALID_ARG
    p = ctypes.c_int64()
    assert L.tw_wave_split(10, 5, 4, None, None, ctypes.byref(p)) == tw.TW_ERR_INVALID_ARG
    opts = tw._SplitOpts(None, 3, 0)  # NULL offsets with a positive count
    assert L.tw_wave_split(10, 5, 4, ctypes.byref(opts), ctypes.byref(p),
                           ctypes.byref(ctypes.c_int64())) == tw.TW_ERR_INVALID_ARG


def test_planner_large_values_no_overflow(L):
    T = 1 << 40
    C = 1 << 30
    p, s = tw.tw_wave_split(T, C, 148)
    assert p + s == T


# ------------------------------------------------------------------ fused-call validation


BASE = 0x7F0000000000  # fake device addresses; validation never dereferences them


def _fused(L, N=2, T=4, H=16, eps=1e-5, sm_budget=0, partials=None, residual=None, gamma=None,
           out=None):
    if partials is None:
        partials = [BASE + (r + 1) * (1 << 24) for r in range(N)]
    arr = (ctypes.c_void_p * max(len(partials), 1))(*partials)
    residual = BASE + (40 << 24) if residual is None else residual
    gamma = BASE + (41 << 24) if gamma is None else gamma
    out = BASE + (42 << 24) if out is None else out
    return L.tw_fused_reduce_residual_rmsnorm(arr, N, residual, gamma, ctypes.c_float(eps), T, H,
                                              out, None, sm_budget)


def test_validation_scalar_args(L):
    assert _fused(L, N=0) == tw.TW_ERR_INVALID_ARG
    assert _fused(L, N=17, partials=[BASE + (r + 1) * (1 << 24) for r in range(17)]) == \
        tw.TW_ERR_INVALID_ARG
    assert _fused(L, T=-1) == tw.TW_ERR_INVALID_ARG
    assert _fused(L, H=0) == tw.TW_ERR_INVALID_ARG
    assert _fused(L, H=12) == tw.TW_ERR_ALIGN
    assert _fused(L, H=tw.TW_MAX_HIDDEN + 8) == tw.TW_ERR_UNSUPPORTED
    assert _fused(L, eps=-1e-5) == tw.TW_ERR_INVALID_ARG
    assert _fused(L, eps=float("nan")) == tw.TW_ERR_INVALID_ARG
    assert _fused(L, eps=float("inf")) == tw.TW_ERR_INVALID_ARG
    assert _fused(L, sm_budget=-1) == tw.TW_ERR_INVALID_ARG
    assert _fused(L, T=1 << 60, H=8192) == tw.TW_ERR_INVALID_ARG


def test_validation_empty_batch_is_a_noop(L):
    # T == 0 returns before looking at pointers or calling CUDA.
    assert _fused(L, T=0, partials=[0, 0], residual=0, gamma=0, out=0) == tw.TW_OK
    arr = (ctypes.c_void_p * 2)(0, 0)
    assert L.tw_run_split(0, arr, 2, None, None, ctypes.c_float(1e-5), 0, 16, None, None, None,
                          0) == tw.TW_OK


def test_validation_pointers(L):
    assert _fused(L, partials=[BASE + (1 << 24), 0]) == tw.TW_ERR_INVALID_ARG
    assert _fused(L, residual=0) == tw.TW_ERR_INVALID_ARG
    assert _fused(L, gamma=0) == tw.TW_ERR_INVALID_ARG
    assert _fused(L, out=0) == tw.TW_ERR_INVALID_ARG
    assert _fused(L, partials=[BASE + (1 << 24) + 8, BASE + (2 << 24)]) == tw.TW_ERR_ALIGN
    assert _fused(L, residual=BASE + (40 << 24) + 4) == tw.TW_ERR_ALIGN
    assert _fused(L, gamma=BASE + (41 << 24) + 2) == tw.TW_ERR_ALIGN
    assert _fused(L, out=BASE + (42 << 24) + 8) == tw.TW_ERR_ALIGN


def test_validation_overlaps(L):
    T, H = 4, 16
    r = BASE + (40 << 24)
    # out overlapping the residual (by one row) is rejected
    assert _fused(L, T=T, H=H, residual=r, out=r + H * 2) == tw.TW_ERR_INVALID_ARG
    # a written tensor partly overlapping a partial or gamma is rejected
    assert _fused(L, T=T, H=H, out=BASE + (1 << 24) + 16) == tw.TW_ERR_INVALID_ARG
    # the residual may not alias a partial, even exactly
    assert _fused(L, T=T, H=H, residual=BASE + (1 << 24)) == tw.TW_ERR_INVALID_ARG
    assert _fused(L, T=T, H=H, residual=BASE + (41 << 24) - 16) == tw.TW_ERR_INVALID_ARG
    # gamma inside a written tensor beyond its first row is rejected too
    # (the residual spans T rows, gamma one row of H values)
    assert _fused(L, T=T, H=H, gamma=r + 2 * H * 2) == tw.TW_ERR_INVALID_ARG
    assert _fused(L, T=T, H=H, gamma=BASE + (42 << 24) + 3 * H * 2) == tw.TW_ERR_INVALID_ARG
    # partials aliasing one another is allowed by validation (reads only):
    # the call gets past validation and fails only at the first CUDA call
    # when there is no GPU, or launches when there is one -- not run here.


def test_run_split_prefix_range(L):
    arr = (ctypes.c_void_p * 2)(BASE + (1 << 24), BASE + (2 << 24))
    for prefix in (-1, 5):
        st = L.tw_run_split(prefix, arr, 2, BASE + (40 << 24), BASE + (41 << 24),
                            ctypes.c_float(1e-5), 4, 16, BASE + (42 << 24), None, None, 0)
        assert st == tw.TW_ERR_INVALID_ARG


def test_launch_shape_validates_before_device_query(L):
    g = ctypes.c_int()
    assert L.tw_launch_shape(4, 12, 2, 0, ctypes.byref(g), None, None, None) == tw.TW_ERR_ALIGN
    assert L.tw_launch_shape(4, 16, 0, 0, ctypes.byref(g), None, None, None) == \
        tw.TW_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(monkeypatch):
    monkeypatch.setattr(tw, "_lib", None)
    monkeypatch.setattr(tw, "LIB_PATH", "/nonexistent/libtw.so")
    with pytest.raises(ImportError):
        tw.lib()


def test_bytes_formula():
    # (N+3) * T * H * 2 + H * 2 : the Llama-3.3-70B layer shape
    assert tw.bytes_per_call(1024, 8192, 8) == 184_565_760
    assert tw.bytes_per_call(128, 4096, 2) == 5_251_072
    assert tw.bytes_per_call(8192, 16384, 8) == 2_952_822_784


def test_split_lookup_table_then_planner(L):
    table = {4096: 2112, 1000: 1000, 7168: 3456}
    assert tw.tw_split_lookup(table, 4096, 256, 148) == (2112, 1984)
    assert tw.tw_split_lookup(table, 1000, 600, 148) == (1000, 0)
    # absent token counts fall back to the wave planner
    for T in (8192, 4864, 1024, 0):
        C = -(-T // 128) * 8
        assert tw.tw_split_lookup(table, T, C, 148) == oplanner.wave_split(T, C, 148)
    assert tw.tw_split_lookup({}, 4864, 304, 148) == (2368, 2496)


def test_split_lookup_rejects_bad_tables(L):
    with pytest.raises(tw.TwError):
        tw.tw_split_lookup({4096: 5000}, 4096, 256, 148)     # prefix beyond T
    with pytest.raises(tw.TwError):
        tw.tw_split_lookup({4096: -1}, 4096, 256, 148)
    p = ctypes.c_int64()
    assert L.tw_split_lookup(None, None, 2, 10, 5, 4, None, ctypes.byref(p),
                             ctypes.byref(ctypes.c_int64())) == tw.TW_ERR_INVALID_ARG
    assert L.tw_split_lookup(None, None, -1, 10, 5, 4, None, ctypes.byref(p),
                             ctypes.byref(ctypes.c_int64())) == tw.TW_ERR_INVALID_ARG


def test_prepared_planner_call_equals_the_planner(L):
    """WaveSplitCall (arguments marshalled once) returns what tw_wave_split
    returns, and what the brute-force oracle returns, for the default grid and
    for every-integer offsets; bad arguments still raise."""
    rng = np.random.default_rng(11)
    for _ in range(200):
        T = int(rng.integers(0, 6000))
        C = int(rng.integers(0, 1200))
        S = int(rng.integers(1, 300))
        w = tw.WaveSplitCall(C, S)
        assert w(T) == tw.tw_wave_split(T, C, S) == oplanner.wave_split(T, C, S)
    w = tw.WaveSplitCall(300, 132, offsets=None, min_split_tokens=0)
    assert w(300) == (132, 168)  # the guide's worked example, in CTA units
    with pytest.raises(tw.TwError):
        tw.WaveSplitCall(10, 0)(100)  # num_sms <= 0


def test_run_wave_split_validates_before_any_cuda_call(L):
    """Plan + run in one call: the fused arguments are checked first, then the
    planner's; an empty batch plans (0, 0) and launches nothing; the plan
    outputs may be NULL. None of these needs a GPU."""
    arr = (ctypes.c_void_p * 2)(0, 0)
    eps = ctypes.c_float(1e-5)
    p, s = ctypes.c_int64(-1), ctypes.c_int64(-1)
    opts = ctypes.byref(tw._opts(tw.DEFAULT_OFFSETS, tw.DEFAULT_MIN_SPLIT_TOKENS)[0])
    f = L.tw_run_wave_split
    assert f(0, 148, opts, arr, 2, None, None, eps, 0, 16, None, None, None, 0,
             ctypes.byref(p), ctypes.byref(s)) == tw.TW_OK
    assert (p.value, s.value) == (0, 0)
    assert f(0, 148, None, arr, 2, None, None, eps, 0, 16, None, None, None, 0, None, None) == tw.TW_OK
    # fused arguments: N out of range, H not a multiple of 8, null pointers (T > 0)
    assert f(8, 148, None, arr, 0, None, None, eps, 4, 16, None, None, None, 0, None, None) == \
        tw.TW_ERR_INVALID_ARG
    assert f(8, 148, None, arr, 2, None, None, eps, 4, 12, None, None, None, 0, None, None) == \
        tw.TW_ERR_ALIGN
    assert f(8, 148, None, arr, 2, None, None, eps, 4, 16, None, None, None, 0, None, None) == \
        tw.TW_ERR_INVALID_ARG
    # planner arguments, checked with valid fused arguments
    for C, S in ((8, 0), (-1, 148)):
        assert f(C, S, None, arr, 2, None, None, eps, 0, 16, None, None, None, 0, None, None) == \
            tw.TW_ERR_INVALID_ARG


def test_binding_rejects_tensors_the_abi_cannot_describe():
    """The C ABI takes raw pointers, so the binding checks what a pointer
    cannot carry: host tensors are refused before any library call."""
    import torch
    P = torch.zeros(2, 4, 16, dtype=torch.bfloat16)
    R = torch.zeros(4, 16, dtype=torch.bfloat16)
    G = torch.ones(16, dtype=torch.bfloat16)
    out = torch.empty_like(R)
    for call in (lambda: tw.tw_fused_reduce_residual_rmsnorm(P, R, G, 1e-5, out),
                 lambda: tw.tw_run_split(2, P, R, G, 1e-5, out),
                 lambda: tw.tw_run_wave_split(8, 148, P, R, G, 1e-5, out),
                 lambda: tw.FusedCall(P, R, G, 1e-5, out),
                 lambda: tw.PlannedSplitCall(8, 148, P, R, G, 1e-5, out),
                 lambda: tw.tw_reduce_partials(P, out),
                 lambda: tw.tw_add_rmsnorm(out, R, G, 1e-5, out)):
        with pytest.raises(ValueError, match="contiguous bf16 CUDA tensor"):
            call()


class _FakeCudaTensor:
    """Stands in for a bf16 CUDA tensor on a given device index: only the
    attributes the binding reads before any library call."""

    def __init__(self, shape, index, ptr=0x10000):
        import torch
        self.shape = torch.Size(shape)
        self.dtype = torch.bfloat16
        self.is_cuda = True
        self.device = torch.device("cuda", index)
        self._ptr = ptr

    def is_contiguous(self):
        return True

    def dim(self):
        return len(self.shape)

    def data_ptr(self):
        return self._ptr

    def get_device(self):
        return self.device.index


class _FakeStream:
    def __init__(self, index):
        import torch
        self.device = torch.device("cuda", index)
        self.cuda_stream = 0


def test_binding_rejects_tensors_on_another_device(monkeypatch):
    """The C ABI launches on the current device and cannot tell which GPU a
    raw pointer belongs to, so the binding refuses any tensor or stream on
    another device before a library call is made."""
    monkeypatch.setattr(tw, "_current_device", lambda: 0)

    def lib_must_not_be_called():
        raise AssertionError("library called before the device check")

    monkeypatch.setattr(tw, "lib", lib_must_not_be_called)
    T, H = 4, 16

    def inputs(bad):
        dev = {name: 1 if name == bad else 0 for name in ("p0", "p1", "R", "G", "out")}
        P = [_FakeCudaTensor((T, H), dev["p0"]), _FakeCudaTensor((T, H), dev["p1"])]
        return (P, _FakeCudaTensor((T, H), dev["R"]), _FakeCudaTensor((H,), dev["G"]),
                _FakeCudaTensor((T, H), dev["out"]))

    for bad in ("p0", "p1", "R", "G", "out"):
        P, R, G, out = inputs(bad)
        for call in (lambda: tw.tw_fused_reduce_residual_rmsnorm(P, R, G, 1e-5, out),
                     lambda: tw.tw_run_split(2, P, R, G, 1e-5, out),
                     lambda: tw.tw_run_wave_split(8, 148, P, R, G, 1e-5, out),
                     lambda: tw.tw_run_split_after(2, P, R, G, 1e-5, out),
                     lambda: tw.FusedCall(P, R, G, 1e-5, out),
                     lambda: tw.SplitCall(P, R, G, 1e-5, out),
                     lambda: tw.PlannedSplitCall(8, 148, P, R, G, 1e-5, out),
                     lambda: tw.UnfusedCall(P, R, G, 1e-5, out)):
            with pytest.raises(ValueError, match="current device is cuda:0"):
                call()
    P, R, G, out = inputs(None)
    with pytest.raises(ValueError, match="current device"):
        tw.tw_reduce_partials([P[0], _FakeCudaTensor((T, H), 1)], out)
    with pytest.raises(ValueError, match="current device"):
        tw.tw_add_rmsnorm(_FakeCudaTensor((T, H), 1), R, G, 1e-5, out)
    # streams on another device
    for call in (lambda: tw.tw_fused_reduce_residual_rmsnorm(P, R, G, 1e-5, out,
                                                             stream=_FakeStream(1)),
                 lambda: tw.tw_run_split(2, P, R, G, 1e-5, out, _FakeStream(0), _FakeStream(1)),
                 lambda: tw.SplitCall(P, R, G, 1e-5, out, _FakeStream(1), _FakeStream(0)),
                 lambda: tw.tw_run_split_after(2, P, R, G, 1e-5, out, stream=_FakeStream(1))):
        with pytest.raises(ValueError, match="stream"):
            call()
