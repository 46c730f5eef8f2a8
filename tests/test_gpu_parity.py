"""Parity of the CUDA path (through the C ABI) with the CPU oracle, and the
bitwise invariants of the launch shape: SM budget, token shards, two-stream
split, repeat runs. Needs a GPU.

Pages cited: [W] "TokenWeave: Why Hiding Tensor-Parallel Communication Needs
Wave Arithmetic, Not Finer Tiles"."""

import math

import numpy as np
import pytest
import torch

import reduce_rmsnorm_gb300 as tw
import synth
from oracle import planner as oplanner
from parity import check_rows, to_gpu

pytestmark = pytest.mark.gpu

EPS = synth.EPS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from reduce_rmsnorm_gb300 import build
    build.build()
    tw.lib()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    tw.tw_device_status(reset=True)
    yield
    assert tw.tw_device_status(reset=True) == 0, "a kernel gave up on a bounded wait"


def run(partials, residual, gamma, eps=EPS, sm_budget=0):
    P, R, G = to_gpu(partials, residual, gamma)
    out = torch.empty_like(R)
    tw.tw_fused_reduce_residual_rmsnorm(P, R, G, eps, out, sm_budget=sm_budget)
    torch.cuda.synchronize()
    return R, out


def assert_same(a, b):
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ------------------------------------------------------------------ parity vs oracle

SMALL = [
    # T, H, N, p_sigma, outliers
    (1, 8, 1, 0.05, 0.0),          # smallest row: one 16-byte vector
    (3, 8, 16, 0.05, 0.0),         # N at its maximum
    (7, 2056, 3, 0.02, 0.0),       # 257 vectors: a one-vector ragged chunk
    (5, 4104, 8, 0.02, 0.0),       # 513 vectors: ragged third chunk
    (9, 2048, 2, 0.05, 0.0),       # exactly one chunk
    (33, 16384, 8, 0.01, 0.01),    # 405B hidden size with outliers
    (2, 32768, 2, 0.02, 0.0),      # hidden size at its maximum (16 chunks)
    (3, 32768, 16, 0.02, 0.0),     # both maxima: 16 partials of 32768
    (300, 1024, 5, 0.02, 0.0),     # more rows than SMs
    (157, 8200, 4, 0.03, 0.0),     # ragged rows and chunks
]


@pytest.mark.parametrize("T,H,N,sig,outl", SMALL)
def test_parity_small(T, H, N, sig, outl):
    p, r, g = synth.make_inputs(T, H, N, sig, outlier_frac=outl, seed=T * 7 + N)
    R, out = run(p, r, g)
    check_rows(p, r, g, EPS, R, out)


def _one_case_per_instance():
    """(H, N) pairs that reach every distinct kernel instance. The launch
    picks VPT = 2 (8 KiB copies) for N <= 8 and VPT = 1 (4 KiB) above; KMAX
    is the smallest power of two >= the row's chunks * VPT; a row is EXACT
    when H / 8 == KMAX * 256. For each KMAX an exact H and a ragged H of the
    same KMAX are paired with every N of the compile-time instances and with
    N that take the runtime-N instance. At one row per CTA, N <= 8 with
    H <= 16384 takes the direct form (its own KMAX: the row's 256-vector
    slots rounded up to a power of two), but for ragged rows over 8192 with
    N >= 6."""
    cases = []
    for exact, ragged in ((2048, 1032), (4096, 2056), (8192, 6152), (16384, 12296),
                          (32768, 24584)):
        for n in range(1, 9):
            cases += [(exact, n), (ragged, n)]
    for exact, ragged in ((2048, 1032), (4096, 3080), (8192, 6152), (16384, 12296),
                          (32768, 24584)):
        for n in (9, 15, 16):
            cases += [(exact, n), (ragged, n)]
    return cases


@pytest.mark.parametrize("T,budget", [(3, 0), (40, 3)])
@pytest.mark.parametrize("H,N", _one_case_per_instance())
def test_parity_every_kernel_instance(H, N, T, budget):
    """T=3: one row per CTA (the direct form for H <= 16384 and N <= 8
    except ragged rows over 8192 with N >= 6, a ring otherwise; the L2 prefetch is issued when the row fits in
    144 KiB); T=40 on 3 SMs: 13-14 rows per CTA, so the ring wraps across
    rows, the prefetch is issued, and KMAX = 4 shapes take the two-pipeline
    forms."""
    p, r, g = synth.make_inputs(T, H, N, 0.02, seed=H + N + T)
    R, out = run(p, r, g, sm_budget=budget)
    check_rows(p, r, g, EPS, R, out)


@pytest.mark.parametrize("eps", [0.0, 1e-6, 1e-5, 0.5])
def test_parity_eps(eps):
    p, r, g = synth.make_inputs(17, 4096, 4, 0.02, seed=5)
    R, out = run(p, r, g, eps=eps)
    check_rows(p, r, g, eps, R, out)


def test_parity_pr1_workload():
    """T=128, H=4096, N=2, P ~ N(0, 0.05^2), R ~ N(0, 1), gamma ~ N(1, 0.1^2)."""
    p, r, g = synth.make_workload("pr1_t128_h4096_n2")
    R, out = run(p, r, g)
    stats = check_rows(p, r, g, EPS, R, out)
    assert stats["rows"] == 128


def test_parity_llama70b_all_rows():
    """T=1024, H=8192, N=8: every row, in the launch the benchmark times."""
    p, r, g = synth.make_workload("llama70b_t1024_h8192_n8")
    P, R, G = to_gpu(p, r, g)
    out = torch.empty_like(R)
    C = math.ceil(1024 / 128) * (8192 // 128) // 8
    step = tw.PlannedSplitCall(C, 148, P, R, G, EPS, out, torch.cuda.current_stream(),
                               torch.cuda.Stream())
    assert step() == (1024, 0)                 # one wave of 64 CTAs: the batch stays whole
    torch.cuda.synchronize()
    stats = check_rows(p, r, g, EPS, R, out)
    assert stats["max_ulp"] <= 2.0


def test_parity_llama405b_sampled_rows():
    """T=8192, H=16384, N=8 with 1% outliers x50: the benchmark's planned call
    at full size, 256 seeded random rows plus the first and last checked
    against the oracle."""
    p, r, g = synth.make_workload("llama405b_t8192_h16384_n8")
    P, R, G = to_gpu(p, r, g)
    out = torch.empty_like(R)
    C = math.ceil(8192 / 128) * (16384 // 128) // 8
    step = tw.PlannedSplitCall(C, 148, P, R, G, EPS, out, torch.cuda.current_stream(),
                               torch.cuda.Stream())
    assert step() == (8192, 0)                 # no offset keeps 1024 CTAs within 7 waves
    torch.cuda.synchronize()
    rng = np.random.Generator(np.random.PCG64(405))
    rows = np.unique(np.concatenate([[0, 8191], rng.choice(8192, 256, replace=False)]))
    check_rows(p, r, g, EPS, R, out, rows=rows)


def test_zero_and_constant_rows():
    T, H, N = 6, 4096, 3
    p, r, g = synth.make_inputs(T, H, N, 0.02, seed=9)
    p[:, 1] = 0
    r[1] = 0                    # zero row -> Y = 0, not NaN
    p[:, 2] = 0
    r[2] = 0.75                 # constant row c -> gamma * c / sqrt(c^2 + eps)
    R, out = run(p, r, g)
    check_rows(p, r, g, EPS, R, out)
    o = out.cpu().float()
    assert torch.all(o[1] == 0)
    want = g.float() * 0.75 / math.sqrt(0.75 ** 2 + EPS)
    assert torch.allclose(o[2], want.to(torch.bfloat16).float(), rtol=2 ** -7, atol=0)


def test_eps_zero_rows_and_the_zero_row():
    """eps = 0 (allowed: eps >= 0). Non-zero rows follow the formula with no
    eps; a row whose z is all zero has no scale, 0 * rsqrt(0), so its Y is
    NaN in every element, as in the formula, while its updated residual is 0."""
    T, H, N = 5, 4096, 2
    p, r, g = synth.make_inputs(T, H, N, 0.02, seed=10)
    p[:, 3] = 0
    r[3] = 0
    R, out = run(p, r, g, eps=0.0)
    keep = [0, 1, 2, 4]
    check_rows(p, r, g, 0.0, R, out, rows=keep)
    assert torch.all(R[3] == 0)
    assert torch.all(torch.isnan(out[3].float()))


def test_subnormal_inputs_are_not_flushed():
    """bf16 subnormals (|x| < 2^-126) in partials and residual: the fp32 sums
    must keep them (no flush to zero), so the updated residual stays bit-exact
    to the IEEE fp32 emulation; rows of only subnormals normalise to tiny
    outputs within tolerance."""
    T, H, N = 8, 2048, 4
    rng = np.random.Generator(np.random.PCG64(126))
    mags = np.ldexp(1.0, rng.integers(-133, -126, size=(N + 1, T, H)))
    vals = mags * rng.choice([-1.0, 1.0], size=(N + 1, T, H)) * rng.integers(1, 128, size=(N + 1, T, H))
    vals[:, :4] = np.where(rng.random((N + 1, 4, H)) < 0.5, vals[:, :4],
                           rng.standard_normal((N + 1, 4, H)) * 1e-3)   # mixed rows
    from oracle import bf16 as obf16
    bits = obf16.encode_rne(vals)
    as_bf16 = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
    p, r = as_bf16[:N].contiguous(), as_bf16[N].contiguous()
    g = synth.make_inputs(1, H, 1, 0.02, seed=5)[2]
    R, out = run(p, r, g)
    check_rows(p, r, g, EPS, R, out)
    b = synth.bits(R.cpu())
    subnormal = ((b & 0x7F80) == 0) & ((b & 0x7F) != 0)
    assert subnormal.any()   # subnormal results were produced


def test_small_integer_partials_exact():
    T, H, N = 4, 1024, 8
    gen = torch.Generator().manual_seed(3)
    p = torch.randint(-4, 5, (N, T, H), generator=gen).to(torch.bfloat16)
    r = torch.randint(-4, 5, (T, H), generator=gen).to(torch.bfloat16)
    g = torch.ones(H, dtype=torch.bfloat16)
    R, out = run(p, r, g)
    want = p.float().sum(0) + r.float()
    assert torch.equal(R.cpu().float(), want)
    check_rows(p, r, g, EPS, R, out)


def test_aliased_partials_allowed():
    T, H = 8, 4096
    p, r, g = synth.make_inputs(T, H, 1, 0.02, seed=4)
    P = p[0].cuda()
    R = r.cuda()
    G = g.cuda()
    out = torch.empty_like(R)
    tw.tw_fused_reduce_residual_rmsnorm([P, P, P], R, G, EPS, out)
    torch.cuda.synchronize()
    check_rows(torch.stack([p[0]] * 3), r, g, EPS, R, out)


def test_inputs_not_modified():
    p, r, g = synth.make_inputs(64, 8192, 8, 0.02, seed=6)
    P, R, G = to_gpu(p, r, g)
    out = torch.empty_like(R)
    tw.tw_fused_reduce_residual_rmsnorm(P, R, G, EPS, out)
    torch.cuda.synchronize()
    assert_same(P.cpu(), p)
    assert_same(G.cpu(), g)


def test_empty_batch():
    H = 4096
    P = torch.empty((2, 0, H), dtype=torch.bfloat16, device="cuda")
    R = torch.empty((0, H), dtype=torch.bfloat16, device="cuda")
    G = torch.ones(H, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(R)
    tw.tw_fused_reduce_residual_rmsnorm(P, R, G, EPS, out)
    torch.cuda.synchronize()


def test_binding_rejects_wrong_dtype_shape_or_strides():
    p, r, g = synth.make_inputs(4, 4096, 2, 0.02)
    P, R, G = to_gpu(p, r, g)
    out = torch.empty_like(R)
    with pytest.raises(ValueError, match="partials"):
        tw.tw_fused_reduce_residual_rmsnorm(P.float(), R, G, EPS, out)       # fp32 partials
    with pytest.raises(ValueError, match="gamma"):
        tw.tw_fused_reduce_residual_rmsnorm(P, R, G[:2048], EPS, out)        # gamma of H/2
    with pytest.raises(ValueError, match="out"):
        tw.tw_fused_reduce_residual_rmsnorm(P, R, G, EPS, out.t())           # transposed view
    with pytest.raises(ValueError, match="partials"):
        tw.tw_fused_reduce_residual_rmsnorm([P[0], P[1][:, :2048]], R, G, EPS, out)  # [T, H/2]
    assert_same(R, to_gpu(p, r, g)[1])                                        # nothing ran


def test_binding_rejects_a_short_or_mistyped_smid_buffer():
    """The debug call writes one int32 per CTA: the binding refuses a buffer
    shorter than the grid, or of another dtype, before any launch."""
    p, r, g = synth.make_inputs(300, 4096, 2, 0.02, seed=4)
    P, R, G = to_gpu(p, r, g)
    out = torch.empty_like(R)
    grid = tw.tw_launch_shape(300, 4096, 2, 0)["grid"]
    for bad in (torch.empty(grid - 1, dtype=torch.int32, device="cuda"),
                torch.empty(grid, dtype=torch.int64, device="cuda"),
                torch.empty(grid, dtype=torch.int32)):
        with pytest.raises(ValueError, match="smid_out"):
            tw.tw_fused_debug_smid(P, R, G, EPS, out, bad)
    assert_same(R, to_gpu(p, r, g)[1])                                        # nothing ran
    smid = torch.full((grid,), -1, dtype=torch.int32, device="cuda")
    tw.tw_fused_debug_smid(P, R, G, EPS, out, smid)
    torch.cuda.synchronize()
    assert min(smid.cpu().tolist()) >= 0


def test_misaligned_pointer_rejected_on_device_tensors():
    p, r, g = synth.make_inputs(4, 4096, 2, 0.02)
    P, R, G = to_gpu(p, r, g)
    flat = torch.empty(4 * 4096 + 8, dtype=torch.bfloat16, device="cuda")
    out = flat[4:4 + 4 * 4096].view(4, 4096)   # 8-byte offset
    with pytest.raises(tw.TwError) as e:
        tw.tw_fused_reduce_residual_rmsnorm(P, R, G, EPS, out)
    assert e.value.status == tw.TW_ERR_ALIGN


# ------------------------------------------------------------------ bitwise invariants


def test_repeat_runs_bitwise():
    p, r, g = synth.make_inputs(200, 8192, 8, 0.02, seed=8)
    a = run(p, r, g)
    b = run(p, r, g)
    assert_same(a[0], b[0])
    assert_same(a[1], b[1])


@pytest.mark.parametrize("budget", [1, 2, 3, 4, 8, 16, 151, 152, 1000])
def test_sm_budget_bitwise(budget):
    p, r, g = synth.make_inputs(1024, 8192, 8, 0.02, seed=1)
    ref = run(p, r, g, sm_budget=0)
    got = run(p, r, g, sm_budget=budget)
    assert_same(ref[0], got[0])
    assert_same(ref[1], got[1])


@pytest.mark.parametrize("H,N", [(8192, 1), (8192, 2), (8192, 3), (8192, 4), (6152, 1),
                                 (6152, 3), (8192, 9), (8192, 12), (8192, 16)])
def test_kernel_forms_bitwise(H, N):
    """The launch picks among kernel forms by speed: one or two pipelines per
    CTA, chunk ring or row ring. Every form must give the same rows bit for
    bit. T = 300 under a 120-SM budget (2.5 rows per CTA, a grid over half
    the SMs) takes the one-pipeline chunk ring; an 8-SM budget takes the
    two-pipeline form for these shapes. The launch shapes are checked to
    differ, so the comparison is between two forms."""
    T = 300
    wide = tw.tw_launch_shape(T, H, N, 120)
    b8 = tw.tw_launch_shape(T, H, N, 8)
    assert wide["threads"] == 288 and b8["threads"] == 544, (wide, b8)
    p, r, g = synth.make_inputs(T, H, N, 0.02, seed=H + 3 * N)
    ref = run(p, r, g, sm_budget=120)
    got = run(p, r, g, sm_budget=8)
    assert_same(ref[0], got[0])
    assert_same(ref[1], got[1])
    rows = [0, 1, 149, 150, 298, 299] + list(range(7, 300, 37))
    check_rows(p, r, g, EPS, got[0], got[1], rows=rows)


def test_shards_bitwise_llama70b():
    """8 token-boundary shards of 128 rows, each launched on its own, equal the
    whole T=1024 batch bit for bit ([W] "Fix two": the norm is per token, so a
    token-boundary shard normalises independently)."""
    p, r, g = synth.make_workload("llama70b_t1024_h8192_n8")
    whole_R, whole_out = run(p, r, g)
    P, R, G = to_gpu(p, r, g)
    out = torch.empty_like(R)
    for s in range(8):
        a, b = s * 128, (s + 1) * 128
        tw.tw_fused_reduce_residual_rmsnorm([P[i, a:b] for i in range(8)], R[a:b], G, EPS, out[a:b])
    torch.cuda.synchronize()
    assert_same(whole_R, R)
    assert_same(whole_out, out)


@pytest.mark.parametrize("T", [1024, 2048, 4096, 8192])
def test_split_configs_bitwise(T):
    """The split workload: plan with 148 SMs and C = ceil(T/128) * 8, run the
    halves on two streams, compare with the unsplit call bit for bit."""
    C = math.ceil(T / 128) * (8192 // 128) // 8
    prefix, suffix = tw.tw_wave_split(T, C, 148)
    assert (prefix, suffix) == oplanner.wave_split(T, C, 148)
    p, r, g = synth.make_inputs(T, 8192, 8, 0.02, seed=T)
    ref = run(p, r, g)
    P, R, G = to_gpu(p, r, g)
    out = torch.empty_like(R)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(sa):
        tw.tw_run_split(prefix, P, R, G, EPS, out, sa, sb)
    sa.synchronize()
    assert_same(ref[0], R)
    assert_same(ref[1], out)
    rng = np.random.Generator(np.random.PCG64(T))
    rows = np.unique(np.concatenate([[0, prefix - 1, prefix, T - 1],
                                     rng.choice(T, 64, replace=False)]))
    rows = rows[(rows >= 0) & (rows < T)]
    check_rows(p, r, g, EPS, R, out, rows=rows)


@pytest.mark.parametrize("prefix", [0, 1, 2368, 4863, 4864])
@pytest.mark.parametrize("budget", [0, 4])
def test_uneven_split_bitwise(prefix, budget):
    T = 4864
    p, r, g = synth.make_inputs(T, 8192, 8, 0.02, seed=48)
    ref = run(p, r, g)
    P, R, G = to_gpu(p, r, g)
    out = torch.empty_like(R)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    tw.tw_run_split(prefix, P, R, G, EPS, out, sa, sb, sm_budget=budget)
    sa.synchronize()
    assert_same(ref[0], R)
    assert_same(ref[1], out)


@pytest.mark.parametrize("T", [128, 4096, 4864])
def test_plan_and_run_in_one_call(T):
    """tw_run_wave_split and the prepared PlannedSplitCall: the plan equals
    the planner's (and the oracle's), and the rows equal the unsplit call's
    bit for bit."""
    C = math.ceil(T / 128) * (8192 // 128) // 8
    plan = oplanner.wave_split(T, C, 148)
    p, r, g = synth.make_inputs(T, 8192, 8, 0.02, seed=T + 3)
    ref = run(p, r, g)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    P, R, G = to_gpu(p, r, g)
    out = torch.empty_like(R)
    assert tw.tw_run_wave_split(C, 148, P, R, G, EPS, out, sa, sb) == plan
    sa.synchronize()
    assert_same(ref[0], R)
    assert_same(ref[1], out)
    P, R, G = to_gpu(p, r, g)
    out = torch.empty_like(R)
    call = tw.PlannedSplitCall(C, 148, P, R, G, EPS, out, sa, sb)
    assert call() == plan
    sa.synchronize()
    assert_same(ref[0], R)
    assert_same(ref[1], out)


def test_split_same_stream():
    T = 300
    p, r, g = synth.make_inputs(T, 4096, 4, 0.02, seed=30)
    ref = run(p, r, g)
    P, R, G = to_gpu(p, r, g)
    out = torch.empty_like(R)
    s = torch.cuda.current_stream()
    tw.tw_run_split(100, P, R, G, EPS, out, s, s)
    torch.cuda.synchronize()
    assert_same(ref[0], R)
    assert_same(ref[1], out)


@pytest.mark.parametrize("N", [8, 2, 12])
@pytest.mark.parametrize("budget", [1, 2, 4, 8, 16])
def test_sm_budget_occupies_at_most_budget_sms(budget, N):
    """N = 8 takes the one-pipeline chunk ring, N = 2 the two-pipeline chunk
    ring and N = 12 the two-pipeline row ring: every form must keep one CTA
    per SM (more than half an SM's shared memory) so that a budget of k CTAs
    occupies at most k SMs."""
    T, H = 512, 8192
    shape = tw.tw_launch_shape(T, H, N, budget)
    assert shape["grid"] == min(budget, T)
    assert shape["smem_bytes"] > 114 * 1024
    assert shape["threads"] == (288 if N == 8 else 544)
    p, r, g = synth.make_inputs(T, H, N, 0.02, seed=2)
    P, R, G = to_gpu(p, r, g)
    out = torch.empty_like(R)
    smid = torch.full((shape["grid"],), -1, dtype=torch.int32, device="cuda")
    tw.tw_fused_debug_smid(P, R, G, EPS, out, smid, sm_budget=budget)
    torch.cuda.synchronize()
    ids = smid.cpu().tolist()
    assert min(ids) >= 0
    assert len(set(ids)) == len(ids) <= budget   # one CTA per SM
    check_rows(p, r, g, EPS, R, out, rows=np.arange(0, T, 37))


def test_full_gpu_one_cta_per_sm():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    shape = tw.tw_launch_shape(4096, 8192, 8, 0)
    assert shape["grid"] == sms
    assert shape["smem_bytes"] > 114 * 1024  # more than half an SM: one CTA per SM
    p, r, g = synth.make_inputs(4096, 8192, 8, 0.02, seed=3)
    P, R, G = to_gpu(p, r, g)
    out = torch.empty_like(R)
    smid = torch.full((sms,), -1, dtype=torch.int32, device="cuda")
    tw.tw_fused_debug_smid(P, R, G, EPS, out, smid)
    torch.cuda.synchronize()
    assert len(set(smid.cpu().tolist())) == sms


def test_offsets_beyond_4gib_sampled_rows():
    """T*H*2 > 2^32 bytes per tensor (T=70000, H=32768, N=1): 64-bit row
    offsets. Inputs are 8 seeded rows tiled over the batch on the device; the
    first, last and a spread of rows are checked against the oracle."""
    T, H, N = 70000, 32768, 1
    base_p, base_r, g = synth.make_inputs(8, H, N, 0.05, seed=70)
    idx = torch.arange(T) % 8
    dev = torch.device("cuda")
    P = base_p.to(dev)[:, idx.to(dev)].contiguous()
    R = base_r.to(dev)[idx.to(dev)].contiguous()
    G = g.to(dev)
    out = torch.empty_like(R)
    torch.cuda.synchronize()
    assert R.numel() * 2 > 2 ** 32
    tw.tw_fused_reduce_residual_rmsnorm(P, R, G, EPS, out)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 7, 8, 32767, 32768, 65535, 65536, 65537, 69990, 69999])
    sel = torch.from_numpy(rows)
    check_rows(base_p[:, sel % 8], base_r[sel % 8], g, EPS, R[sel.to(dev)].cpu(),
               out[sel.to(dev)].cpu())
    del P, R, out
    torch.cuda.empty_cache()


def test_split_runner_captured_in_cuda_graph():
    """tw_run_split captured into a CUDA graph (fork and join become graph
    edges) replays to bitwise the same result as the eager unsplit call."""
    T = 4096
    C = math.ceil(T / 128) * 8
    prefix = tw.tw_wave_split(T, C, 148)[0]
    assert 0 < prefix < T
    p, r, g = synth.make_inputs(T, 8192, 8, 0.02, seed=44)
    ref = run(p, r, g)
    P, R, G = to_gpu(p, r, g)
    R0 = R.clone()
    out = torch.empty_like(R)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    sa.wait_stream(torch.cuda.current_stream())
    call = tw.SplitCall(P, R, G, EPS, out, sa, sb)
    with torch.cuda.stream(sa):
        call(prefix)                      # eager first: attributes and events exist
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=sa):
        call(prefix)
    for _ in range(2):
        R.copy_(R0)
        out.zero_()
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert_same(ref[0], R)
        assert_same(ref[1], out)


def _random_shapes(count, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    shapes = []
    while len(shapes) < count:
        H = 8 * int(rng.integers(1, 4097))
        N = int(rng.integers(1, 17))
        T = int(rng.integers(1, 400))
        if T * H * (N + 1) > 3_000_000:     # keep the oracle to seconds
            continue
        budget = int(rng.choice([0, 0, 1, 3, 7, 33]))
        shapes.append((T, H, N, budget))
    return shapes


@pytest.mark.parametrize("T,H,N,budget", _random_shapes(24, 2026))
def test_parity_random_shapes(T, H, N, budget):
    """Seeded random shapes: any hidden size that is a multiple of 8 (ragged
    chunks), 1..16 partials, ragged row counts, SM budgets; every row checked."""
    p, r, g = synth.make_inputs(T, H, N, 0.03, seed=T + H + N)
    R, out = run(p, r, g, sm_budget=budget)
    check_rows(p, r, g, EPS, R, out)


def _random_two_pipeline_shapes(count, seed):
    """Shapes that take the two-pipeline forms: H/8 in 513..1024 with
    N = 1..4 (the chunk ring; ragged H only up to N = 3), or H = 8192 with
    N = 9..16 (the row ring), under budgets where every CTA owns >= 4 rows."""
    rng = np.random.Generator(np.random.PCG64(seed))
    shapes = []
    while len(shapes) < count:
        budget = int(rng.choice([2, 3, 5, 8]))
        if rng.random() < 0.5:
            N = int(rng.integers(1, 5))
            H = 8 * int(rng.integers(513, 1025)) if N <= 3 else 8192
        else:
            N, H = int(rng.integers(9, 17)), 8192
        T = int(rng.integers(4 * budget, 4 * budget + 60))
        if T * H * (N + 1) > 8_000_000:     # keep the oracle to seconds
            continue
        shapes.append((T, H, N, budget))
    return shapes


@pytest.mark.parametrize("T,H,N,budget", _random_two_pipeline_shapes(16, 77))
def test_parity_random_two_pipeline_shapes(T, H, N, budget):
    """Seeded random shapes in the two-pipeline forms, every row checked
    against the oracle, and bitwise equal to the whole-GPU launch of the same
    rows. There every CTA owns one row: the direct form for N <= 8, the
    one-pipeline chunk ring otherwise."""
    shape = tw.tw_launch_shape(T, H, N, budget)
    assert shape["threads"] == 544, (T, H, N, budget, shape)
    assert tw.tw_launch_shape(T, H, N, 0)["threads"] == (256 if _takes_direct(H, N) else 288)
    p, r, g = synth.make_inputs(T, H, N, 0.03, seed=T + H + N + budget)
    R, out = run(p, r, g, sm_budget=budget)
    check_rows(p, r, g, EPS, R, out)
    R1, out1 = run(p, r, g, sm_budget=0)
    assert_same(R, R1)
    assert_same(out, out1)


@pytest.mark.parametrize("T", [1, 16, 76])
@pytest.mark.parametrize("N", [9, 16])
def test_one_row_per_cta_takes_the_chunk_ring(T, N):
    """N >= 9 at H = 8192 with one row per CTA: the one-pipeline chunk ring,
    with every source's chunks in flight, rather than the two-pipeline row
    ring (one of whose pipelines would idle). Every row against the oracle, and
    bitwise equal to a 4-SM budget launch (the row ring once a CTA owns more
    than one row)."""
    H = 8192
    assert tw.tw_launch_shape(T, H, N, 0)["threads"] == 288
    assert tw.tw_launch_shape(T, H, N, 4)["threads"] == (288 if T <= 4 else 544)
    p, r, g = synth.make_inputs(T, H, N, 0.02, seed=7 * T + N)
    R, out = run(p, r, g)
    check_rows(p, r, g, EPS, R, out)
    R4, out4 = run(p, r, g, sm_budget=4)
    assert_same(R, R4)
    assert_same(out, out4)


def _takes_direct(H, N):
    """The direct form's domain at one row per CTA: N <= 8 and at most 8
    slots of 256 vectors, except ragged rows of 5-8 slots with N >= 6 (those
    instances spilled and are not built)."""
    slots = -(-(H // 8) // 256)
    kmax = 1 << (slots - 1).bit_length()
    exact = H // 8 == kmax * 256
    return N <= 8 and kmax <= 8 and not (kmax == 8 and not exact and N >= 6)


@pytest.mark.parametrize("H", [2048, 4096, 8192, 16384, 1032, 5120, 12296])
@pytest.mark.parametrize("N", [1, 3, 5, 8])
def test_direct_form_against_the_ring_and_the_oracle(H, N):
    """One row per CTA with N <= 8 and H <= 16384 takes the direct form (no
    producer warp, no shared-memory ring), whole-slot rows (H = 2048, 4096,
    8192, 16384) and ragged ones alike, except ragged rows over 8192 with
    N >= 6. T = 152 on the whole GPU against the same rows under an 8-SM
    budget (19 rows per CTA: a ring form) bit for bit, and every row against
    the oracle."""
    T = 152
    full = tw.tw_launch_shape(T, H, N, 0)
    if _takes_direct(H, N):
        assert (full["threads"], full["smem_bytes"], full["stages"]) == (256, 0, 0), full
    else:
        assert full["threads"] == 288 and full["smem_bytes"] > 0, full
    assert tw.tw_launch_shape(T, H, N, 8)["smem_bytes"] > 0
    p, r, g = synth.make_inputs(T, H, N, 0.02, outlier_frac=0.01, seed=H + 11 * N)
    R, out = run(p, r, g)
    check_rows(p, r, g, EPS, R, out)
    R8, out8 = run(p, r, g, sm_budget=8)
    assert_same(R, R8)
    assert_same(out, out8)


@pytest.mark.parametrize("T,H,N", [(160, 4096, 8), (256, 4096, 2), (304, 8192, 4),
                                   (200, 6144, 2), (300, 16384, 2), (256, 8192, 8),
                                   (305, 4096, 8), (608, 4096, 4), (760, 4096, 2),
                                   (761, 4096, 2), (456, 8192, 2)])
def test_one_cta_per_row_while_the_rows_fit_at_once(T, H, N):
    """On the whole GPU with more rows than SMs: one direct-form CTA per row
    while all of them fit on the GPU at once (k CTAs per SM by their
    registers: 5 at H = 4096, N = 2; 4 at N = 4; 2 at N = 8; 1 at H = 8192,
    N = 8), a ring CTA per SM otherwise. Every row against the oracle, and
    bit for bit against the same rows under an 8-SM budget (a ring form)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    shape = tw.tw_launch_shape(T, H, N, 0)
    direct = shape["threads"] == 256
    assert shape["grid"] == (T if direct else min(T, sms)), shape
    if (T, H, N) in ((160, 4096, 8), (608, 4096, 4), (760, 4096, 2)):
        assert direct
    if (T, H, N) in ((256, 8192, 8), (305, 4096, 8), (761, 4096, 2)):
        assert not direct
    p, r, g = synth.make_inputs(T, H, N, 0.02, seed=T + H + N)
    R, out = run(p, r, g)
    check_rows(p, r, g, EPS, R, out)
    R8, out8 = run(p, r, g, sm_budget=8)
    assert_same(R, R8)
    assert_same(out, out8)


@pytest.mark.parametrize("T", [1, 7, 100])
def test_direct_form_output_over_a_partial_and_smid(T):
    """The direct form with Y written over partial 5, against Y into its own
    buffer; and its %smid record names a valid SM for every CTA."""
    H, N = 8192, 8
    p, r, g = synth.make_inputs(T, H, N, 0.02, seed=300 + T)
    ref = run(p, r, g)
    P, R, G = to_gpu(p, r, g)
    out = P[5]
    tw.tw_fused_reduce_residual_rmsnorm(P, R, G, EPS, out)
    torch.cuda.synchronize()
    assert_same(ref[0], R)
    assert_same(ref[1], out)
    P, R, G = to_gpu(p, r, g)
    out = torch.empty_like(R)
    smid = torch.full((T,), -1, dtype=torch.int32, device="cuda")
    tw.tw_fused_debug_smid(P, R, G, EPS, out, smid)
    torch.cuda.synchronize()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert int(smid.min()) >= 0 and int(smid.max()) < sms
    assert_same(ref[1], out)


@pytest.mark.parametrize("which,budget,split,N", [(0, 0, False, 8), (7, 0, False, 8),
                                                   (3, 4, False, 8), (0, 0, True, 8),
                                                   (1, 8, False, 2), (11, 8, False, 12)])
def test_output_written_over_a_partial(which, budget, split, N):
    """out == partials[r]: Y written over one rank's partial equals the result
    into a separate buffer, bit for bit (also under an SM budget and split,
    and in the two-pipeline chunk ring (N=2) and row ring (N=12))."""
    T, H = 2048, 8192
    p, r, g = synth.make_inputs(T, H, N, 0.02, seed=91)
    ref = run(p, r, g, sm_budget=budget)
    P, R, G = to_gpu(p, r, g)
    out = P[which]
    if split:
        sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
        tw.tw_run_split(T // 2 + 64, P, R, G, EPS, out, sa, sb, sm_budget=budget)
    else:
        tw.tw_fused_reduce_residual_rmsnorm(P, R, G, EPS, out, sm_budget=budget)
    torch.cuda.synchronize()
    assert_same(ref[0], R)
    assert_same(ref[1], out)
