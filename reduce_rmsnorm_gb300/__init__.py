"""Python binding of libtw: fused reduce + residual + RMSNorm on one GB300.

Argument marshalling only. Every step of the computation runs in libtw's CUDA
kernels (``csrc/``) behind the C ABI declared in ``include/tw.h``; PyTorch
supplies device memory and streams. There is no fallback: if ``libtw.so`` is
missing or a call fails, an exception is raised.

The functions carry the C names:

    tw_fused_reduce_residual_rmsnorm(partials, residual, gamma, eps, out, stream=None, sm_budget=0)
    tw_wave_split(num_tokens, ctas_unsplit, num_sms, offsets=DEFAULT_OFFSETS, min_split_tokens=1024)
    tw_split_lookup(table, num_tokens, ctas_unsplit, num_sms, offsets=..., min_split_tokens=...)
    tw_run_split(prefix_tokens, partials, residual, gamma, eps, out, stream_a, stream_b, sm_budget=0)
    tw_run_wave_split(ctas_unsplit, num_sms, partials, residual, gamma, eps, out, stream_a, stream_b,
                      sm_budget=0, offsets=..., min_split_tokens=...)          # plan + run
    tw_run_split_after(prefix_tokens, partials, residual, gamma, eps, out, stream,
                       prefix_ready, suffix_ready, sm_budget=0)
    tw_strerror(status)
    tw_launch_shape(T, H, N, sm_budget=0)
    tw_device_status(reset=True)
    tw_fused_debug_smid(partials, residual, gamma, eps, out, smid_out, stream=None, sm_budget=0)
    tw_reduce_partials(partials, sum_out, stream=None)                 # unfused baseline
    tw_add_rmsnorm(sum_in, residual, gamma, eps, out, stream=None)     # unfused baseline
    tw_shard_rows(num_tokens, world, rank)                              # token-boundary shard

The token-shard form of the step across tensor-parallel ranks (all-to-all,
fused step on the rank's shard, all-gather) is ``shard.TokenShardStep``.

For launch-bound loops, ``FusedCall``, ``SplitCall``, ``WaveSplitCall`` and
``PlannedSplitCall`` marshal the arguments once and then make a single ctypes
call each time they are called.
"""

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtw.so")

TW_OK = 0
TW_ERR_INVALID_ARG = 1
TW_ERR_ALIGN = 2
TW_ERR_UNSUPPORTED = 3
TW_ERR_CUDA = 4
TW_ERR_DEVICE = 5
TW_MAX_PARTIALS = 16
TW_MAX_HIDDEN = 32768

DEFAULT_OFFSETS = (0, 64, 128, 192, 256, 512)
DEFAULT_MIN_SPLIT_TOKENS = 1024

EXPORTED = ("tw_fused_reduce_residual_rmsnorm", "tw_wave_split", "tw_run_split", "tw_strerror",
            "tw_launch_shape", "tw_device_status", "tw_fused_debug_smid", "tw_reduce_partials",
            "tw_add_rmsnorm", "tw_run_split_after", "tw_split_lookup", "tw_debug_wait_timeout",
            "tw_run_wave_split", "tw_shard_rows")


class TwError(RuntimeError):
    """A libtw call returned a status other than TW_OK."""

    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s" % (where, tw_strerror(status)))


class _SplitOpts(ctypes.Structure):
    _fields_ = [("offsets", ctypes.POINTER(ctypes.c_int)), ("n_offsets", ctypes.c_int),
                ("min_split_tokens", ctypes.c_int)]


_lib = None
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int


def lib():
    """The loaded libtw (ctypes.CDLL). Raises ImportError if it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError("libtw.so is not built (%s); run `python -m reduce_rmsnorm_gb300.build`"
                          % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    L.tw_fused_reduce_residual_rmsnorm.argtypes = [ctypes.POINTER(_vp), _int, _vp, _vp,
                                                   ctypes.c_float, _i64, _i64, _vp, _vp, _int]
    L.tw_fused_reduce_residual_rmsnorm.restype = _int
    L.tw_fused_debug_smid.argtypes = [ctypes.POINTER(_vp), _int, _vp, _vp, ctypes.c_float, _i64,
                                      _i64, _vp, _vp, _int, _vp]
    L.tw_fused_debug_smid.restype = _int
    L.tw_wave_split.argtypes = [_i64, _i64, _int, ctypes.POINTER(_SplitOpts),
                                ctypes.POINTER(_i64), ctypes.POINTER(_i64)]
    L.tw_wave_split.restype = _int
    L.tw_debug_wait_timeout.argtypes = [_i64, _vp]
    L.tw_debug_wait_timeout.restype = _int
    L.tw_split_lookup.argtypes = [ctypes.POINTER(_i64), ctypes.POINTER(_i64), _int, _i64, _i64,
                                  _int, ctypes.POINTER(_SplitOpts), ctypes.POINTER(_i64),
                                  ctypes.POINTER(_i64)]
    L.tw_split_lookup.restype = _int
    L.tw_run_split.argtypes = [_i64, ctypes.POINTER(_vp), _int, _vp, _vp, ctypes.c_float, _i64,
                               _i64, _vp, _vp, _vp, _int]
    L.tw_run_split.restype = _int
    L.tw_run_wave_split.argtypes = [_i64, _int, ctypes.POINTER(_SplitOpts), ctypes.POINTER(_vp),
                                    _int, _vp, _vp, ctypes.c_float, _i64, _i64, _vp, _vp, _vp,
                                    _int, ctypes.POINTER(_i64), ctypes.POINTER(_i64)]
    L.tw_run_wave_split.restype = _int
    L.tw_strerror.argtypes = [_int]
    L.tw_strerror.restype = ctypes.c_char_p
    L.tw_launch_shape.argtypes = [_i64, _i64, _int, _int] + [ctypes.POINTER(_int)] * 4
    L.tw_launch_shape.restype = _int
    L.tw_device_status.argtypes = [_int, ctypes.POINTER(_int)]
    L.tw_device_status.restype = _int
    L.tw_run_split_after.argtypes = [_i64, ctypes.POINTER(_vp), _int, _vp, _vp, ctypes.c_float,
                                     _i64, _i64, _vp, _vp, _vp, _vp, _int]
    L.tw_run_split_after.restype = _int
    L.tw_reduce_partials.argtypes = [ctypes.POINTER(_vp), _int, _i64, _i64, _vp, _vp]
    L.tw_reduce_partials.restype = _int
    L.tw_add_rmsnorm.argtypes = [_vp, _vp, _vp, ctypes.c_float, _i64, _i64, _vp, _vp]
    L.tw_add_rmsnorm.restype = _int
    L.tw_shard_rows.argtypes = [_i64, _int, _int, ctypes.POINTER(_i64), ctypes.POINTER(_i64)]
    L.tw_shard_rows.restype = _int
    _lib = L
    return L


def _check(status, where):
    if status != TW_OK:
        raise TwError(status, where)


def tw_strerror(status):
    return lib().tw_strerror(int(status)).decode()


# ------------------------------------------------------------------ marshalling helpers


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _partials_array(partials):
    """Host array of device pointers from a list of tensors or an [N, T, H] tensor."""
    import torch
    if isinstance(partials, torch.Tensor):
        seq = [partials[i] for i in range(partials.shape[0])] if partials.dim() == 3 else [partials]
    else:
        seq = list(partials)
    arr = (_vp * max(len(seq), 1))(*[t.data_ptr() for t in seq])
    return arr, len(seq)


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _shape(residual):
    if residual.dim() != 2:
        raise ValueError("residual must be [T, H]")
    return int(residual.shape[0]), int(residual.shape[1])


_BF16 = None


def _bad_tensor(t, name, shape):
    import torch
    if not isinstance(t, torch.Tensor):
        return TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        return ValueError("%s must be a contiguous bf16 CUDA tensor (got %s, %s, contiguous=%s)"
                          % (name, t.dtype, t.device, t.is_contiguous()))
    return ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


def _check_tensor(t, name, shape):
    """A bf16, contiguous CUDA tensor of the given shape: the layout the C ABI
    takes as a raw pointer (it cannot see dtypes or strides)."""
    global _BF16
    if _BF16 is None:
        import torch
        _BF16 = torch.bfloat16
    try:
        ok = t.dtype is _BF16 and t.is_cuda and t.is_contiguous() and t.shape == shape
    except AttributeError:
        ok = False
    if not ok:
        raise _bad_tensor(t, name, shape)


def _current_device():
    """Index of the CUDA device current on this thread: the device the C ABI
    launches on (it calls cudaGetDevice)."""
    import torch
    return torch.cuda.current_device()


def _check_devices(where, tensors=(), streams=()):
    """Every tensor and stream must be on the current device. The C ABI
    launches on the current device and cannot tell from a raw pointer which
    GPU owns it: another GPU's address would reach the kernel's bulk copies
    and stores as a peer access, or fault. Streams given as raw handles
    (ints) cannot be checked here."""
    dev = _current_device()
    for name, t in tensors:
        if t is not None and t.get_device() != dev:
            raise ValueError("%s: %s is on %s but the current device is cuda:%d; all tensors "
                             "and streams must be on the current device" % (where, name, t.device,
                                                                            dev))
    for name, s in streams:
        d = getattr(s, "device", None)
        if d is not None and d.index != dev:
            raise ValueError("%s: %s is on %s but the current device is cuda:%d; all tensors "
                             "and streams must be on the current device" % (where, name, d, dev))


def _step_args(partials, residual, gamma, out, where="fused step", streams=()):
    """Validated (pointer array, N, T, H) for a fused step's tensors. An
    [N, T, H] stack is checked once and its N pointers are computed from its
    base address and stride. Every tensor and stream must be on the current
    device (_check_devices)."""
    import torch
    T, H = _shape(residual)
    _check_tensor(residual, "residual", (T, H))
    _check_tensor(gamma, "gamma", (H,))
    _check_tensor(out, "out", (T, H))
    named = [("residual", residual), ("gamma", gamma), ("out", out)]
    if isinstance(partials, torch.Tensor) and partials.dim() == 3:
        n = int(partials.shape[0])
        if not (partials.dtype is torch.bfloat16 and partials.is_cuda and
                tuple(partials.shape[1:]) == (T, H) and
                (T * H == 0 or (partials.stride(2) == 1 and (T <= 1 or partials.stride(1) == H)))):
            raise ValueError("partials must be [N, %d, %d] bf16 CUDA with contiguous [T, H] "
                             "slices (got %s, %s, shape %s, strides %s)"
                             % (T, H, partials.dtype, partials.device, tuple(partials.shape),
                                partials.stride()))
        _check_devices(where, named + [("partials", partials)], streams)
        base, step = partials.data_ptr(), partials.stride(0) * 2
        return (_vp * max(n, 1))(*[base + i * step for i in range(n)]), n, T, H
    seq = [partials] if isinstance(partials, torch.Tensor) else list(partials)
    for r, t in enumerate(seq):
        _check_tensor(t, "partials[%d]" % r, (T, H))
    _check_devices(where, named + [("partials[%d]" % r, t) for r, t in enumerate(seq)], streams)
    arr, n = _partials_array(seq)
    return arr, n, T, H


# ------------------------------------------------------------------ entry points


def tw_fused_reduce_residual_rmsnorm(partials, residual, gamma, eps, out, stream=None, sm_budget=0):
    """Fused step over rows [0, T): residual <- bf16(sum P + R); out <- RMSNorm.

    partials: list of N bf16 [T, H] CUDA tensors or one [N, T, H] tensor;
    residual (in/out), out: bf16 [T, H]; gamma: bf16 [H]. Shapes are read from
    ``residual``; layout and error rules are those of the C call.
    """
    arr, n, T, H = _step_args(partials, residual, gamma, out, "tw_fused_reduce_residual_rmsnorm",
                              [("stream", stream)])
    st = lib().tw_fused_reduce_residual_rmsnorm(arr, n, _ptr(residual), _ptr(gamma), float(eps), T,
                                                H, _ptr(out), _stream(stream), int(sm_budget))
    _check(st, "tw_fused_reduce_residual_rmsnorm")


def tw_fused_debug_smid(partials, residual, gamma, eps, out, smid_out, stream=None, sm_budget=0):
    """The fused call that also records each CTA's SM id into ``smid_out``: a
    contiguous int32 CUDA tensor with at least the launch grid's length
    (``tw_launch_shape(T, H, N, sm_budget)["grid"]``). The kernel writes one
    entry per CTA, so a shorter buffer is refused here, before any launch."""
    import torch
    arr, n, T, H = _step_args(partials, residual, gamma, out, "tw_fused_debug_smid",
                              [("stream", stream)])
    grid = tw_launch_shape(T, H, n, sm_budget)["grid"] if T > 0 else 0
    if not (isinstance(smid_out, torch.Tensor) and smid_out.dtype is torch.int32 and
            smid_out.is_cuda and smid_out.is_contiguous() and smid_out.numel() >= grid):
        raise ValueError("smid_out must be a contiguous int32 CUDA tensor with at least %d "
                         "entries (the launch grid)" % grid)
    _check_devices("tw_fused_debug_smid", [("smid_out", smid_out)])
    st = lib().tw_fused_debug_smid(arr, n, _ptr(residual), _ptr(gamma), float(eps), T, H, _ptr(out),
                                   _stream(stream), int(sm_budget), _ptr(smid_out))
    _check(st, "tw_fused_debug_smid")


def _opts_arg(offsets, min_split_tokens):
    """(options pointer, objects to keep alive) for the C planner. The pages'
    defaults go as NULL, which the planner serves from its own static list."""
    if (offsets is DEFAULT_OFFSETS or (offsets is not None and
                                       tuple(offsets) == tuple(DEFAULT_OFFSETS))) and \
            min_split_tokens == DEFAULT_MIN_SPLIT_TOKENS:
        return None, None
    opts, keep = _opts(offsets, min_split_tokens)
    return ctypes.byref(opts), (opts, keep)


def tw_wave_split(num_tokens, ctas_unsplit, num_sms, offsets=DEFAULT_OFFSETS,
                  min_split_tokens=DEFAULT_MIN_SPLIT_TOKENS):
    """(prefix_tokens, suffix_tokens) of the wave-aware split.

    offsets=None means every integer offset 0 .. half-1.
    """
    optp, keep = _opts_arg(offsets, min_split_tokens)
    p, s = _i64(), _i64()
    st = lib().tw_wave_split(int(num_tokens), int(ctas_unsplit), int(num_sms), optp,
                             ctypes.byref(p), ctypes.byref(s))
    del keep
    _check(st, "tw_wave_split")
    return p.value, s.value


def _opts(offsets, min_split_tokens):
    if offsets is None:
        return _SplitOpts(None, 0, int(min_split_tokens)), None
    keep = (ctypes.c_int * max(len(offsets), 1))(*[int(o) for o in offsets])
    return _SplitOpts(keep, len(offsets), int(min_split_tokens)), keep


def tw_split_lookup(table, num_tokens, ctas_unsplit, num_sms, offsets=DEFAULT_OFFSETS,
                    min_split_tokens=DEFAULT_MIN_SPLIT_TOKENS):
    """(prefix, suffix) from ``table`` ({token count: prefix}) if it has the
    token count, else from tw_wave_split."""
    items = sorted(table.items())
    toks = (_i64 * max(len(items), 1))(*[int(k) for k, _ in items])
    pref = (_i64 * max(len(items), 1))(*[int(v) for _, v in items])
    optp, keep = _opts_arg(offsets, min_split_tokens)
    p, s = _i64(), _i64()
    st = lib().tw_split_lookup(toks, pref, len(items), int(num_tokens), int(ctas_unsplit),
                               int(num_sms), optp, ctypes.byref(p), ctypes.byref(s))
    del keep
    _check(st, "tw_split_lookup")
    return p.value, s.value


def tw_run_split(prefix_tokens, partials, residual, gamma, eps, out, stream_a=None, stream_b=None,
                 sm_budget=0):
    """Rows [0, prefix) on stream_a, [prefix, T) on stream_b; stream_a joins both."""
    arr, n, T, H = _step_args(partials, residual, gamma, out, "tw_run_split",
                              [("stream_a", stream_a), ("stream_b", stream_b)])
    st = lib().tw_run_split(int(prefix_tokens), arr, n, _ptr(residual), _ptr(gamma), float(eps), T,
                            H, _ptr(out), _stream(stream_a), _stream(stream_b), int(sm_budget))
    _check(st, "tw_run_split")


def tw_run_wave_split(ctas_unsplit, num_sms, partials, residual, gamma, eps, out,
                      stream_a=None, stream_b=None, sm_budget=0, offsets=DEFAULT_OFFSETS,
                      min_split_tokens=DEFAULT_MIN_SPLIT_TOKENS):
    """The wave-aware plan and the split step in one C call; returns the plan
    (prefix_tokens, suffix_tokens)."""
    arr, n, T, H = _step_args(partials, residual, gamma, out, "tw_run_wave_split",
                              [("stream_a", stream_a), ("stream_b", stream_b)])
    optp, keep = _opts_arg(offsets, min_split_tokens)
    p, s = _i64(), _i64()
    st = lib().tw_run_wave_split(int(ctas_unsplit), int(num_sms), optp, arr, n,
                                 _ptr(residual), _ptr(gamma), float(eps), T, H, _ptr(out),
                                 _stream(stream_a), _stream(stream_b), int(sm_budget),
                                 ctypes.byref(p), ctypes.byref(s))
    del keep
    _check(st, "tw_run_wave_split")
    return p.value, s.value


def tw_shard_rows(num_tokens, world, rank):
    """(row0, rows) of `rank`'s token-boundary shard of a num_tokens batch
    over `world` ranks: contiguous shards of ceil(T / world) rows in rank
    order, the tail shorter."""
    a, b = _i64(), _i64()
    _check(lib().tw_shard_rows(int(num_tokens), int(world), int(rank), ctypes.byref(a),
                               ctypes.byref(b)), "tw_shard_rows")
    return a.value, b.value


def _event(e):
    return None if e is None else ctypes.c_void_p(e.cuda_event if hasattr(e, "cuda_event") else int(e))


def tw_run_split_after(prefix_tokens, partials, residual, gamma, eps, out, stream=None,
                       prefix_ready=None, suffix_ready=None, sm_budget=0):
    """On `stream`: wait prefix_ready, fused step on rows [0, prefix); wait
    suffix_ready, fused step on rows [prefix, T). Events: torch.cuda.Event or
    raw cudaEvent_t handles."""
    arr, n, T, H = _step_args(partials, residual, gamma, out, "tw_run_split_after",
                              [("stream", stream)])
    st = lib().tw_run_split_after(int(prefix_tokens), arr, n, _ptr(residual), _ptr(gamma),
                                  float(eps), T, H, _ptr(out), _stream(stream),
                                  _event(prefix_ready), _event(suffix_ready), int(sm_budget))
    _check(st, "tw_run_split_after")


def tw_reduce_partials(partials, sum_out, stream=None):
    """Unfused baseline, kernel 1: sum_out <- bf16(sum of the partials)."""
    T, H = _shape(sum_out)
    _check_tensor(sum_out, "sum_out", (T, H))
    seq = [partials[i] for i in range(partials.shape[0])] if hasattr(partials, "dim") and \
        partials.dim() == 3 else list(partials)
    for r, t in enumerate(seq):
        _check_tensor(t, "partials[%d]" % r, (T, H))
    _check_devices("tw_reduce_partials", [("sum_out", sum_out)] +
                   [("partials[%d]" % r, t) for r, t in enumerate(seq)], [("stream", stream)])
    arr, n = _partials_array(seq)
    st = lib().tw_reduce_partials(arr, n, T, H, _ptr(sum_out), _stream(stream))
    _check(st, "tw_reduce_partials")


def tw_add_rmsnorm(sum_in, residual, gamma, eps, out, stream=None):
    """Unfused baseline, kernel 2: residual <- bf16(sum + residual); out <- RMSNorm(residual)."""
    T, H = _shape(residual)
    for name, t, shape in (("sum_in", sum_in, (T, H)), ("residual", residual, (T, H)),
                           ("gamma", gamma, (H,)), ("out", out, (T, H))):
        _check_tensor(t, name, shape)
    _check_devices("tw_add_rmsnorm", [("sum_in", sum_in), ("residual", residual),
                                      ("gamma", gamma), ("out", out)], [("stream", stream)])
    st = lib().tw_add_rmsnorm(_ptr(sum_in), _ptr(residual), _ptr(gamma), float(eps), T, H,
                              _ptr(out), _stream(stream))
    _check(st, "tw_add_rmsnorm")


class FusedCall:
    """tw_fused_reduce_residual_rmsnorm with its arguments marshalled once.

    Holds references to the tensors; calling the object launches the step on
    the stream resolved at construction."""

    def __init__(self, partials, residual, gamma, eps, out, stream=None, sm_budget=0):
        arr, n, T, H = _step_args(partials, residual, gamma, out, "FusedCall", [("stream", stream)])
        self.tensors = (partials, residual, gamma, out)
        self._fn = lib().tw_fused_reduce_residual_rmsnorm
        self._args = (arr, _int(n), _ptr(residual), _ptr(gamma), ctypes.c_float(eps), _i64(T),
                      _i64(H), _ptr(out), _stream(stream), _int(int(sm_budget)))

    def __call__(self):
        st = self._fn(*self._args)
        if st != TW_OK:
            raise TwError(st, "tw_fused_reduce_residual_rmsnorm")


class WaveSplitCall:
    """tw_wave_split for fixed (ctas_unsplit, num_sms, options), marshalled
    once: calling it with a token count returns (prefix_tokens,
    suffix_tokens). The plan is still computed by the C planner on every
    call."""

    def __init__(self, ctas_unsplit, num_sms, offsets=DEFAULT_OFFSETS,
                 min_split_tokens=DEFAULT_MIN_SPLIT_TOKENS):
        optp, self._keep = _opts_arg(offsets, min_split_tokens)
        self._p, self._s = _i64(), _i64()
        self._fn = lib().tw_wave_split
        self._tail = (_i64(int(ctas_unsplit)), _int(int(num_sms)), optp,
                      ctypes.byref(self._p), ctypes.byref(self._s))

    def __call__(self, num_tokens):
        st = self._fn(int(num_tokens), *self._tail)
        if st != TW_OK:
            raise TwError(st, "tw_wave_split")
        return self._p.value, self._s.value


class SplitCall:
    """tw_run_split with its arguments marshalled once; call it with the
    prefix token count."""

    def __init__(self, partials, residual, gamma, eps, out, stream_a=None, stream_b=None,
                 sm_budget=0):
        arr, n, T, H = _step_args(partials, residual, gamma, out, "SplitCall",
                                  [("stream_a", stream_a), ("stream_b", stream_b)])
        self.tokens = T
        self.tensors = (partials, residual, gamma, out)
        self._fn = lib().tw_run_split
        self._args = (arr, _int(n), _ptr(residual), _ptr(gamma), ctypes.c_float(eps), _i64(T),
                      _i64(H), _ptr(out), _stream(stream_a), _stream(stream_b),
                      _int(int(sm_budget)))

    def __call__(self, prefix_tokens):
        st = self._fn(int(prefix_tokens), *self._args)
        if st != TW_OK:
            raise TwError(st, "tw_run_split")


class PlannedSplitCall:
    """tw_run_wave_split with its arguments marshalled once: each call plans
    the split in C (the planner runs every time) and runs the step; it
    returns the plan (prefix_tokens, suffix_tokens)."""

    def __init__(self, ctas_unsplit, num_sms, partials, residual, gamma, eps, out,
                 stream_a=None, stream_b=None, sm_budget=0, offsets=DEFAULT_OFFSETS,
                 min_split_tokens=DEFAULT_MIN_SPLIT_TOKENS):
        arr, n, T, H = _step_args(partials, residual, gamma, out, "PlannedSplitCall",
                                  [("stream_a", stream_a), ("stream_b", stream_b)])
        self.tokens = T
        self.tensors = (partials, residual, gamma, out)
        optp, self._keep = _opts_arg(offsets, min_split_tokens)
        self._p, self._s = _i64(), _i64()
        self._fn = lib().tw_run_wave_split
        self._args = (_i64(int(ctas_unsplit)), _int(int(num_sms)), optp, arr,
                      _int(n), _ptr(residual), _ptr(gamma), ctypes.c_float(eps), _i64(T), _i64(H),
                      _ptr(out), _stream(stream_a), _stream(stream_b), _int(int(sm_budget)),
                      ctypes.byref(self._p), ctypes.byref(self._s))

    def __call__(self):
        st = self._fn(*self._args)
        if st != TW_OK:
            raise TwError(st, "tw_run_wave_split")
        return self._p.value, self._s.value


class UnfusedCall:
    """The unfused baseline with its arguments marshalled once: calling it
    launches tw_reduce_partials into ``out`` and then tw_add_rmsnorm over
    ``out`` in place (two launches)."""

    def __init__(self, partials, residual, gamma, eps, out, stream=None):
        arr, n, T, H = _step_args(partials, residual, gamma, out, "UnfusedCall",
                                  [("stream", stream)])
        self.tensors = (partials, residual, gamma, out)
        L = lib()
        s = _stream(stream)
        self._reduce = (L.tw_reduce_partials, (arr, n, T, H, _ptr(out), s))
        self._norm = (L.tw_add_rmsnorm, (_ptr(out), _ptr(residual), _ptr(gamma),
                                         ctypes.c_float(eps), T, H, _ptr(out), s))

    def __call__(self):
        for fn, args in (self._reduce, self._norm):
            st = fn(*args)
            if st != TW_OK:
                raise TwError(st, fn.__name__)


def tw_launch_shape(T, H, N, sm_budget=0):
    """dict(grid, threads, smem_bytes, stages) of the launch on the current device."""
    g, t, m, s = _int(), _int(), _int(), _int()
    st = lib().tw_launch_shape(int(T), int(H), int(N), int(sm_budget), ctypes.byref(g),
                               ctypes.byref(t), ctypes.byref(m), ctypes.byref(s))
    _check(st, "tw_launch_shape")
    return dict(grid=g.value, threads=t.value, smem_bytes=m.value, stages=s.value)


def tw_debug_wait_timeout(limit_ns, stream=None):
    """Diagnostic: a bounded wait that runs out after limit_ns (sets the error word)."""
    _check(lib().tw_debug_wait_timeout(int(limit_ns), _stream(stream)), "tw_debug_wait_timeout")


def tw_device_status(reset=True):
    """The device error word (0 = no kernel gave up a wait); synchronises."""
    code = _int()
    _check(lib().tw_device_status(1 if reset else 0, ctypes.byref(code)), "tw_device_status")
    return code.value


def bytes_per_call(T, H, N):
    """Algorithmic HBM bytes of one fused call: read N partials and the
    residual, write the residual and the output, read gamma once."""
    return (N + 3) * T * H * 2 + H * 2
