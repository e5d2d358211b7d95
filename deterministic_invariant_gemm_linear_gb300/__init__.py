"""Deterministic, batch-invariant BF16 contractions for GB300 (sm_103a).

A thin ctypes binding over the C ABI in ``include/rlk.h`` (librlk.so, built
in-tree by ``build.py``).  This module only marshals arguments: PyTorch is used
for device memory and streams; every step of every operator runs in the
library's CUDA kernels.  There is no CPU or PyTorch fallback — if the library
is missing, or the device is not sm_103, calls raise.

Operators (web pages of the RL-Kernel project):
  * ``linear_logp`` — "feat(linear-logp): add batch-invariant fused SM90
    operator": log_softmax(hidden . W^T + bias)[target] and the log-sum-exp,
    with a vocabulary split that depends on V only.  Forward only: inputs that
    require grad are rejected (the page's author notes: backward is outside
    the contract and fails closed).
  * ``det_gemm_fwd / det_gemm_da / det_gemm_db`` — "feat(musa): add native
    deterministic gemm kernel": C = A B, dA = dC B^T, dB = A^T dC with FP32
    accumulation in a fixed ascending K order, BF16 or FP32 output; an FP32 dC
    is rounded to BF16 first (that page's review comment).
  * ``linear_logp_trainable``, ``det_gemm_trainable``, ``det_linear_trainable`` —
    opt-in torch.autograd wiring of the forward entries to the library's
    backward entries (gradients bitwise equal to calling those entries).
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
# RLK_LIBRARY=debug selects the debug build (store checks, phase trace) of the
# same library; anything else, or unset, the release build.
LIB_PATH = os.path.join(_PKG_DIR, "librlk_debug.so" if os.environ.get("RLK_LIBRARY") == "debug"
                        else "librlk.so")

RLK_OK = 0
RLK_BF16, RLK_FP32 = 0, 1
RLK_GEMM_FWD, RLK_GEMM_DA, RLK_GEMM_DB = 0, 1, 2
RLK_GEMM_LINEAR_FWD, RLK_GEMM_LINEAR_DX, RLK_GEMM_LINEAR_DW, RLK_GEMM_FWD_ACCUM = 3, 4, 5, 6
STATUS_NAMES = {0: "RLK_OK", 1: "RLK_ERR_NULL", 2: "RLK_ERR_SHAPE", 3: "RLK_ERR_DTYPE",
                4: "RLK_ERR_ALIGN", 5: "RLK_ERR_WORKSPACE", 6: "RLK_ERR_UNSUPPORTED_DEVICE",
                7: "RLK_ERR_CUDA", 8: "RLK_ERR_TIMEOUT", 9: "RLK_ERR_BOUNDS",
                10: "RLK_ERR_NOT_DEBUG_BUILD"}
RLK_DEVERR_TIMEOUT, RLK_DEVERR_BOUNDS = 0x1, 0x2
TRACE_FIELDS, TRACE_MAX_CTAS = 16, 1024


class RlkError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


_P, _I64, _SZ, _I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int

# name -> (restype, argtypes); mirrors include/rlk.h
SIGNATURES = {
    "rlk_status_string": (ctypes.c_char_p, [_I]),
    "rlk_numerics_version": (_I, []),
    "rlk_device_check": (_I, []),
    "rlk_get_device_error": (_I, [_P, ctypes.POINTER(ctypes.c_uint32)]),
    "rlk_selftest_bounded_wait": (_I, [ctypes.c_uint32, _P]),
    "rlk_is_debug_build": (_I, []),
    "rlk_selftest_store_check": (_I, [_P]),
    "rlk_debug_trace_read": (_I, [_P, _I64, ctypes.POINTER(_I64)]),
    "rlk_vocab_split_policy": (_I, [_I64, ctypes.POINTER(_I64), ctypes.POINTER(_I64),
                                    ctypes.POINTER(_I64)]),
    "rlk_linear_logp_workspace_size": (_SZ, [_P, _I64, _I64, _I64, _P, _I64, _I64]),
    "rlk_linear_logp": (_I, [_P, _I64, _I64, _I64, _P, _I64, _I64, _P, _P, _I64,
                             _P, _P, _P, _P, _SZ, _P]),
    "rlk_linear_logp_partials": (_I, [_P, _I64, _I64, _I64, _P, _I64, _I64, _P, _P, _I64,
                                      _P, _SZ, _P]),
    "rlk_linear_logp_combine": (_I, [_I64, _I64, _P, _I64, _P, _P, _P, _P, _SZ, _P]),
    "rlk_linear_logp_noalloc": (_I, [_P, _I64, _I64, _I64, _P, _I64, _I64, _P, _P, _I64,
                                     _P, _P, _P, _P]),
    "rlk_throughput_split_count": (_I, [_I64, _I64, ctypes.c_int32, ctypes.POINTER(_I64)]),
    "rlk_det_gemm_tile_plan": (_I, [_I, _I64, _I64, _I64, ctypes.c_int32,
                                    ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(_I64),
                                    ctypes.POINTER(ctypes.c_int32)]),
    "rlk_vocab_shard_range": (_I, [_I64, _I64, _I64, ctypes.POINTER(_I64), ctypes.POINTER(_I64),
                                   ctypes.POINTER(_I64), ctypes.POINTER(_I64)]),
    "rlk_linear_logp_shard_workspace_size": (_SZ, [_P, _I64, _I64, _I64, _P, _I64, _I64, _I64,
                                                   _I64]),
    "rlk_linear_logp_shard_partials": (_I, [_P, _I64, _I64, _I64, _P, _I64, _I64, _I64, _I64, _P,
                                            _P, _I64, _P, _I64, _P, _P, _SZ, _P]),
    "rlk_linear_logp_combine_shards": (_I, [_I64, _I64, _P, _I64, _I64, _P, _P, _I64, _I64, _P,
                                            _I64, _P, _P, _P, _P]),
    "rlk_linear_logp_splits_workspace_size": (_SZ, [_P, _I64, _I64, _I64, _P, _I64, _I64, _I64]),
    "rlk_linear_logp_splits": (_I, [_P, _I64, _I64, _I64, _P, _I64, _I64, _P, _P, _I64,
                                    _P, _P, _P, _I64, _P, _SZ, _P]),
    "rlk_linear_logp_backward_workspace_size": (_SZ, [_I64, _I64]),
    "rlk_linear_logp_backward_workspace_size_for": (_SZ, [_P, _I64, _I64, _I64, _P, _I64, _I64]),
    "rlk_linear_logp_backward": (_I, [_P, _I64, _I64, _I64, _P, _I64, _I64, _P, _P, _I64, _P, _P,
                                      _P, _I, _I64, _P, _I, _I64, _P, _P, _SZ, _P]),
    "rlk_det_gemm_workspace_size": (_SZ, [_I, _P, _I, _I64, _I64, _I64, _P, _I, _I64, _I64, _I64]),
    "rlk_det_gemm_fwd": (_I, [_P, _I64, _I64, _I64, _P, _I64, _I64, _P, _I, _I64, _P, _SZ, _P]),
    "rlk_det_gemm_da": (_I, [_P, _I, _I64, _I64, _I64, _P, _I64, _I64, _P, _I, _I64, _P, _SZ, _P]),
    "rlk_det_gemm_db": (_I, [_P, _I64, _I64, _I64, _P, _I, _I64, _I64, _P, _I, _I64, _P, _SZ, _P]),
    "rlk_det_gemm_fwd_accum_fp32": (_I, [_P, _I64, _I64, _I64, _P, _I64, _I64, _P, _I64, _P, _SZ,
                                         _P]),
    "rlk_sum_partials_ordered": (_I, [_P, _I64, _I64, _I64, _I64, _I64, _P, _I, _I64, _P]),
    "rlk_det_linear_fwd": (_I, [_P, _I64, _I64, _I64, _P, _I64, _I64, _P, _I, _I64, _P, _SZ, _P]),
    "rlk_det_linear_dx": (_I, [_P, _I, _I64, _I64, _I64, _P, _I64, _I64, _P, _I, _I64, _P, _SZ, _P]),
    "rlk_det_linear_dw": (_I, [_P, _I, _I64, _I64, _I64, _P, _I64, _I64, _P, _I, _I64, _P, _SZ, _P]),
    "rlk_det_gemm_backward_workspace_size": (_SZ, [_P, _I, _I64, _I64, _I64, _P, _I64, _I64, _P,
                                                   _I64]),
    "rlk_det_gemm_backward": (_I, [_P, _I, _I64, _I64, _I64, _P, _I64, _I64, _P, _I64, _P, _I,
                                   _I64, _P, _I, _I64, _P, _SZ, _P]),
    "rlk_det_linear_backward_workspace_size": (_SZ, [_P, _I, _I64, _I64, _I64, _P, _I64, _I64, _P,
                                                     _I64]),
    "rlk_det_linear_backward": (_I, [_P, _I, _I64, _I64, _I64, _P, _I64, _I64, _P, _I64, _P, _I,
                                     _I64, _P, _I, _I64, _P, _SZ, _P]),
}

_LIB = None


def lib() -> ctypes.CDLL:
    """The loaded librlk.so; raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"librlk.so is not built ({LIB_PATH}); build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        cdll = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(cdll, name)
            f.restype = res
            f.argtypes = args
        _LIB = cdll
    return _LIB


def status_string(status: int) -> str:
    return lib().rlk_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != RLK_OK:
        raise RlkError(status, what)


def numerics_version() -> int:
    return int(lib().rlk_numerics_version())


def vocab_split_policy(V: int):
    """(num_splits, vtiles_per_split, num_vtiles) for a vocabulary of V ids."""
    s, v, t = _I64(), _I64(), _I64()
    _check(lib().rlk_vocab_split_policy(V, ctypes.byref(s), ctypes.byref(v), ctypes.byref(t)),
           "rlk_vocab_split_policy")
    return s.value, v.value, t.value


def device_error(stream=None) -> int:
    """Reads and clears the library's device error word (synchronises the stream)."""
    flags = ctypes.c_uint32(0)
    st = lib().rlk_get_device_error(_stream_ptr(stream), ctypes.byref(flags))
    if st not in (RLK_OK, 8, 9):
        _check(st, "rlk_get_device_error")
    return flags.value


def is_debug_build() -> bool:
    return bool(lib().rlk_is_debug_build())


def debug_trace(max_ctas: int = TRACE_MAX_CTAS):
    """Debug build: the linear-logp kernels' per-CTA phase timestamps (ns) since the
    last read, as a list of TRACE_FIELDS-tuples indexed by CTA (then cleared)."""
    import numpy as np
    out = np.zeros((max_ctas, TRACE_FIELDS), dtype=np.uint64)
    n = _I64()
    _check(lib().rlk_debug_trace_read(out.ctypes.data_as(ctypes.c_void_p), max_ctas,
                                      ctypes.byref(n)), "rlk_debug_trace_read")
    return out[:n.value]


def _stream_ptr(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _matrix(t: torch.Tensor, name: str):
    """(tensor, leading dimension) for a 2-D row-major operand (unit column stride)."""
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D, got shape {tuple(t.shape)}")
    if t.stride(1) != 1 or (t.size(0) > 1 and t.stride(0) < t.size(1)):
        t = t.contiguous()
    ld = t.stride(0) if t.size(0) > 1 else max(t.size(1), t.stride(0))
    return t, ld


def _require_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("rlk operates on CUDA tensors only (no CPU fallback)")


_DT = {torch.bfloat16: RLK_BF16, torch.float32: RLK_FP32}


# ------------------------------------------------------------------ linear-logp
def linear_logp_workspace(hidden2d, weight, ldh, ldw, N, H, V) -> torch.Tensor:
    n = lib().rlk_linear_logp_workspace_size(_ptr(hidden2d), N, H, ldh, _ptr(weight), V, ldw)
    if n == 0 and N > 0:
        raise RlkError(2, "rlk_linear_logp_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=hidden2d.device)


def throughput_split_count(N: int, V: int, sm_count: int = 0) -> int:
    """The occupancy-driven split count of the throughput-mode ablation (depends on N)."""
    s = _I64()
    _check(lib().rlk_throughput_split_count(N, V, sm_count, ctypes.byref(s)),
           "rlk_throughput_split_count")
    return s.value


def det_gemm_tile_plan(op: int, out_rows: int, out_cols: int, red: int, sm_count: int) -> dict:
    """The output tiling of det_gemm op (RLK_GEMM_*) for these extents on sm_count SMs
    (host arithmetic): {"tile_cols": 256 | 224 | 128, "split_blocks": wide blocks run as
    halves, "launches": 1 | 2}."""
    t, b, n = ctypes.c_int32(), _I64(), ctypes.c_int32()
    _check(lib().rlk_det_gemm_tile_plan(op, out_rows, out_cols, red, sm_count, ctypes.byref(t),
                                        ctypes.byref(b), ctypes.byref(n)), "rlk_det_gemm_tile_plan")
    return {"tile_cols": t.value, "split_blocks": b.value, "launches": n.value}


def linear_logp(hidden: torch.Tensor, weight: torch.Tensor, target: torch.Tensor,
                bias: torch.Tensor | None = None, *, return_target_logit: bool = False,
                stream=None, num_splits: int | None = None):
    """logp, lse (FP32, shaped like hidden's leading dims) [, target logit].

    hidden [..., H] bf16, weight [V, H] bf16, target [...] int64 (any strides,
    including an expanded zero-stride target), bias [V] fp32 or None.
    num_splits (ablation only): an explicit vocabulary split count instead of
    the V-only policy (rlk_linear_logp_splits); 0 means the V-only policy.
    """
    if hidden.requires_grad or weight.requires_grad or (bias is not None and bias.requires_grad):
        raise RuntimeError("linear_logp is forward-only: inputs that require grad are rejected")
    _require_cuda(hidden, weight, target, bias)
    if hidden.dtype != torch.bfloat16 or weight.dtype != torch.bfloat16:
        raise TypeError("hidden and weight must be bfloat16")
    if target.dtype != torch.int64:
        raise TypeError("target must be int64")
    if bias is not None and (bias.dtype != torch.float32 or bias.dim() != 1):
        raise TypeError("bias must be a 1-D float32 tensor")
    lead = hidden.shape[:-1]
    H = hidden.size(-1)
    h2, ldh = _matrix(hidden.reshape(-1, H), "hidden")
    w2, ldw = _matrix(weight, "weight")
    N, V = h2.size(0), w2.size(0)
    if w2.size(1) != H:
        raise ValueError("weight must be [V, H] with the hidden size H")
    t1 = target.reshape(-1)
    if t1.numel() != N:
        raise ValueError("target must have one id per hidden row")
    tstride = t1.stride(0) if N > 1 else 1
    if bias is not None:
        bias = bias.contiguous()
        if bias.numel() != V:
            raise ValueError("bias must have V entries")
    dev = hidden.device
    logp = torch.empty(N, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    zt = torch.empty(N, dtype=torch.float32, device=dev) if return_target_logit else None
    with torch.cuda.device(dev):
        if num_splits is None:
            ws = linear_logp_workspace(h2, w2, ldh, ldw, N, H, V)
            st = lib().rlk_linear_logp(_ptr(h2), N, H, ldh, _ptr(w2), V, ldw, _ptr(bias), _ptr(t1),
                                       tstride, _ptr(logp), _ptr(lse), _ptr(zt), _ptr(ws),
                                       ws.numel(), _stream_ptr(stream))
        else:
            n = lib().rlk_linear_logp_splits_workspace_size(_ptr(h2), N, H, ldh, _ptr(w2), V, ldw,
                                                            num_splits)
            if n == 0 and N > 0:
                raise RlkError(2, "rlk_linear_logp_splits_workspace_size")
            ws = torch.empty(n, dtype=torch.uint8, device=dev)
            st = lib().rlk_linear_logp_splits(_ptr(h2), N, H, ldh, _ptr(w2), V, ldw, _ptr(bias),
                                              _ptr(t1), tstride, _ptr(logp), _ptr(lse), _ptr(zt),
                                              num_splits, _ptr(ws), ws.numel(),
                                              _stream_ptr(stream))
    _check(st, "rlk_linear_logp")
    out = (logp.reshape(lead), lse.reshape(lead))
    if return_target_logit:
        out = out + (zt.reshape(lead),)
    return out


class LinearLogpCall:
    """A prepared linear-logp call on fixed tensors (outputs and workspace
    allocated once), runnable as the whole operator or as its two stages."""

    def __init__(self, hidden, weight, target, bias=None, *, target_logit: bool = False,
                 num_splits: int | None = None):
        _require_cuda(hidden, weight, target, bias)
        self.num_splits = num_splits      # None: the operator; an int: the ablation entry point
        self.h, self.ldh = _matrix(hidden, "hidden")
        self.w, self.ldw = _matrix(weight, "weight")
        self.t = target.reshape(-1)
        self.bias = None if bias is None else bias.contiguous()
        self.N, self.H = self.h.shape
        self.V = self.w.size(0)
        self.tstride = self.t.stride(0) if self.N > 1 else 1
        dev = hidden.device
        self.logp = torch.empty(self.N, dtype=torch.float32, device=dev)
        self.lse = torch.empty(self.N, dtype=torch.float32, device=dev)
        self.zt = torch.empty(self.N, dtype=torch.float32, device=dev) if target_logit else None
        with torch.cuda.device(dev):
            if num_splits is None:
                self.ws = linear_logp_workspace(self.h, self.w, self.ldh, self.ldw, self.N, self.H,
                                                self.V)
            else:
                n = lib().rlk_linear_logp_splits_workspace_size(
                    _ptr(self.h), self.N, self.H, self.ldh, _ptr(self.w), self.V, self.ldw,
                    num_splits)
                if n == 0 and self.N > 0:
                    raise RlkError(2, "rlk_linear_logp_splits_workspace_size")
                self.ws = torch.empty(n, dtype=torch.uint8, device=dev)

    def partials(self, stream=None):
        if self.num_splits is not None:
            raise RuntimeError("the two-stage calls use the V-only split")
        _check(lib().rlk_linear_logp_partials(
            _ptr(self.h), self.N, self.H, self.ldh, _ptr(self.w), self.V, self.ldw, _ptr(self.bias),
            _ptr(self.t), self.tstride, _ptr(self.ws), self.ws.numel(), _stream_ptr(stream)),
            "rlk_linear_logp_partials")

    def combine(self, stream=None):
        if self.num_splits is not None:
            raise RuntimeError("the two-stage calls use the V-only split")
        _check(lib().rlk_linear_logp_combine(
            self.N, self.V, _ptr(self.t), self.tstride, _ptr(self.logp), _ptr(self.lse),
            _ptr(self.zt), _ptr(self.ws), self.ws.numel(), _stream_ptr(stream)),
            "rlk_linear_logp_combine")

    def __call__(self, stream=None):
        if self.num_splits is None:
            _check(lib().rlk_linear_logp(
                _ptr(self.h), self.N, self.H, self.ldh, _ptr(self.w), self.V, self.ldw,
                _ptr(self.bias), _ptr(self.t), self.tstride, _ptr(self.logp), _ptr(self.lse),
                _ptr(self.zt), _ptr(self.ws), self.ws.numel(), _stream_ptr(stream)),
                "rlk_linear_logp")
        else:
            _check(lib().rlk_linear_logp_splits(
                _ptr(self.h), self.N, self.H, self.ldh, _ptr(self.w), self.V, self.ldw,
                _ptr(self.bias), _ptr(self.t), self.tstride, _ptr(self.logp), _ptr(self.lse),
                _ptr(self.zt), self.num_splits, _ptr(self.ws), self.ws.numel(),
                _stream_ptr(stream)), "rlk_linear_logp_splits")
        return self.logp, self.lse


# ------------------------------------------------------------ vocabulary shards
def vocab_shard_range(V: int, num_shards: int, shard: int):
    """(split_begin, split_end, v_begin, v_end) of shard `shard` in the balanced
    partition of the V-only splits into num_shards contiguous runs."""
    out = [_I64() for _ in range(4)]
    _check(lib().rlk_vocab_shard_range(V, num_shards, shard, *[ctypes.byref(x) for x in out]),
           "rlk_vocab_shard_range")
    return tuple(x.value for x in out)


def linear_logp_shard_partials(hidden: torch.Tensor, weight_shard: torch.Tensor,
                               target: torch.Tensor, V: int, split_begin: int, split_end: int,
                               bias_shard: torch.Tensor | None = None, *, ld_partials: int = 0,
                               stream=None):
    """Partials of one vocabulary shard: (partials [N, ld, 2] fp32 with the shard's
    (m, s) pairs in its first split_end - split_begin columns, target logits [N]
    fp32, NaN for rows whose target the shard does not hold).

    weight_shard [v_end - v_begin, H] bf16 holds the weight rows of the shard's
    vocabulary ids, bias_shard the matching bias entries; V is the whole
    vocabulary; target holds global ids.
    """
    _require_cuda(hidden, weight_shard, target, bias_shard)
    h2, ldh = _matrix(hidden.reshape(-1, hidden.size(-1)), "hidden")
    w2, ldw = _matrix(weight_shard, "weight_shard")
    N, H = h2.shape
    t1 = target.reshape(-1)
    tstride = t1.stride(0) if N > 1 else 1
    n = split_end - split_begin
    ld = max(ld_partials, n, 1)
    if bias_shard is not None:
        bias_shard = bias_shard.contiguous()
    dev = hidden.device
    partials = torch.empty(N, ld, 2, dtype=torch.float32, device=dev)
    zt = torch.full((N,), float("nan"), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        nb = lib().rlk_linear_logp_shard_workspace_size(_ptr(h2), N, H, ldh, _ptr(w2), V,
                                                        split_begin, split_end, ldw)
        if nb == 0:
            raise RlkError(2, "rlk_linear_logp_shard_workspace_size")
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        _check(lib().rlk_linear_logp_shard_partials(
            _ptr(h2), N, H, ldh, _ptr(w2), V, split_begin, split_end, ldw, _ptr(bias_shard),
            _ptr(t1), tstride, _ptr(partials), ld, _ptr(zt), _ptr(ws), nb, _stream_ptr(stream)),
            "rlk_linear_logp_shard_partials")
    return partials, zt


def linear_logp_combine_shards(partials: torch.Tensor, target_logits: torch.Tensor,
                               split_offsets, target: torch.Tensor, V: int, *,
                               return_target_logit: bool = False, stream=None):
    """The fixed-order merge over gathered shard outputs.

    partials [R, N, ld, 2] fp32 (shard q's pairs in its first
    split_offsets[q+1] - split_offsets[q] columns), target_logits [R, N] fp32,
    split_offsets R + 1 split indices (0 .. S).  Returns logp, lse [, target logit],
    bitwise equal to linear_logp on the whole vocabulary.
    """
    _require_cuda(partials, target_logits, target)
    if partials.dim() != 4 or partials.size(-1) != 2 or partials.dtype != torch.float32:
        raise ValueError("partials must be a float32 [R, N, ld, 2] tensor")
    partials = partials.contiguous()
    target_logits = target_logits.contiguous()
    R, N, ld, _ = partials.shape
    if len(split_offsets) != R + 1:
        raise ValueError("split_offsets needs one entry per shard plus one")
    if tuple(target_logits.shape) != (R, N):
        raise ValueError("target_logits must be [R, N] like the partials' first two dims")
    offs = (ctypes.c_int64 * (R + 1))(*[int(x) for x in split_offsets])
    t1 = target.reshape(-1)
    tstride = t1.stride(0) if N > 1 else 1
    dev = partials.device
    logp = torch.empty(N, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    zt = torch.empty(N, dtype=torch.float32, device=dev) if return_target_logit else None
    with torch.cuda.device(dev):
        _check(lib().rlk_linear_logp_combine_shards(
            N, V, _ptr(t1), tstride, R, offs, _ptr(partials), ld, N * ld, _ptr(target_logits), N,
            _ptr(logp), _ptr(lse), _ptr(zt), _stream_ptr(stream)), "rlk_linear_logp_combine_shards")
    return (logp, lse, zt) if return_target_logit else (logp, lse)


def _all_gather(t: torch.Tensor, group=None) -> torch.Tensor:
    """Every rank's equally shaped tensor, stacked in rank order on t's device.
    With the NCCL backend device tensors are exchanged directly; with gloo they
    travel through host copies."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    dev = t.device
    x = t.contiguous()
    if dist.get_backend(group) != "nccl":
        x = x.cpu()
    parts = [torch.empty_like(x) for _ in range(world)]
    dist.all_gather(parts, x, group=group)
    return torch.stack(parts).to(dev)


def exchange_shard_partials(partials: torch.Tensor, target_logit: torch.Tensor, group=None):
    """All-gather every rank's shard output: ([R, N, ld, 2], [R, N]) in rank order.

    Every rank passes partials padded to the same [N, ld, 2] (the widest shard).
    With the NCCL backend the device tensors are exchanged directly; with gloo the
    tensors travel through host copies and come back on the caller's device.
    """
    return _all_gather(partials, group), _all_gather(target_logit, group)


def sum_partials_ordered(parts: torch.Tensor, out_dtype=torch.float32, *, stream=None):
    """out = parts[0] + parts[1] + ... (FP32, ascending part order) for parts [P, rows, cols]
    fp32, written as out_dtype (bf16 rounds to nearest even)."""
    _require_cuda(parts)
    if parts.dim() != 3 or parts.dtype != torch.float32:
        raise ValueError("parts must be a float32 [P, rows, cols] tensor")
    parts = parts.contiguous()
    P, rows, cols = parts.shape
    out = torch.empty(rows, cols, dtype=out_dtype, device=parts.device)
    with torch.cuda.device(parts.device):
        _check(lib().rlk_sum_partials_ordered(_ptr(parts), P, rows, cols, cols, rows * cols,
                                              _ptr(out), _DT[out_dtype], cols, _stream_ptr(stream)),
               "rlk_sum_partials_ordered")
    return out


def det_gemm_db_row_sharded(A_local: torch.Tensor, dC_local: torch.Tensor,
                            out_dtype=torch.bfloat16, *, group=None):
    """dB = A^T . dC when the rows of A and dC are divided between the ranks of `group`:
    each rank forms its FP32 partial product (det_gemm_db over its own rows), the ranks
    all-gather the partials, and every rank adds them in rank order
    (sum_partials_ordered).  The result is the same bits on every rank and run to
    run; it depends on the row partition, not on the exchange."""
    local = det_gemm_db(A_local, dC_local, out_dtype=torch.float32)
    return sum_partials_ordered(_all_gather(local, group), out_dtype)


def vocab_parallel_linear_logp(hidden: torch.Tensor, weight_shard: torch.Tensor,
                               target: torch.Tensor, V: int,
                               bias_shard: torch.Tensor | None = None, *, group=None,
                               return_target_logit: bool = False):
    """linear_logp with the vocabulary divided between the ranks of `group`.

    Rank q holds the weight rows (and bias entries) of its balanced shard,
    vocab_shard_range(V, world, q); every rank passes the same hidden and target.
    Each rank computes its shard's partials, the ranks exchange them
    (exchange_shard_partials), and every rank merges all of them in the fixed
    order: the results equal single-device linear_logp bit for bit.
    """
    import torch.distributed as dist
    world, rank = dist.get_world_size(group), dist.get_rank(group)
    ranges = [vocab_shard_range(V, world, q) for q in range(world)]
    j0, j1, v0, v1 = ranges[rank]
    if weight_shard.size(0) != v1 - v0:
        raise ValueError(f"rank {rank} holds vocabulary ids [{v0}, {v1}): weight_shard needs "
                         f"{v1 - v0} rows, got {weight_shard.size(0)}")
    widest = max(r[1] - r[0] for r in ranges)
    partials, zt = linear_logp_shard_partials(hidden, weight_shard, target, V, j0, j1, bias_shard,
                                              ld_partials=widest)
    gp, gz = exchange_shard_partials(partials, zt, group)
    offsets = [r[0] for r in ranges] + [ranges[-1][1]]
    out = linear_logp_combine_shards(gp, gz, offsets, target, V,
                                     return_target_logit=return_target_logit)
    lead = hidden.shape[:-1]
    return tuple(o.reshape(lead) for o in out)


def linear_logp_backward(hidden: torch.Tensor, weight: torch.Tensor, target: torch.Tensor,
                         lse: torch.Tensor, grad_logp: torch.Tensor, bias: torch.Tensor | None = None,
                         *, grad_hidden: bool = True, grad_weight: bool = True,
                         grad_bias: bool | None = None, out_dtype=torch.bfloat16,
                         return_grad_logits: bool = False, stream=None):
    """(grad_hidden [..., H], grad_weight [V, H], grad_bias [V] | None) for logp = linear_logp(...).

    lse is the forward's lse; grad_logp is dL/dlogp (same leading shape as hidden's rows).
    With return_grad_logits, also returns G = dL/dz as the BF16 [N, V] view the kernels used.
    """
    _require_cuda(hidden, weight, target, lse, grad_logp, bias)
    lead = hidden.shape[:-1]
    H = hidden.size(-1)
    h2, ldh = _matrix(hidden.reshape(-1, H), "hidden")
    w2, ldw = _matrix(weight, "weight")
    N, V = h2.size(0), w2.size(0)
    t1 = target.reshape(-1)
    tstride = t1.stride(0) if N > 1 else 1
    l1 = lse.reshape(-1).contiguous().float()
    g1 = grad_logp.reshape(-1).contiguous().float()
    if bias is not None:
        bias = bias.contiguous()
    if grad_bias is None:
        grad_bias = bias is not None
    dev = hidden.device
    gh = torch.empty(N, H, dtype=out_dtype, device=dev) if grad_hidden else None
    gw = torch.empty(V, H, dtype=out_dtype, device=dev) if grad_weight else None
    gb = torch.empty(V, dtype=torch.float32, device=dev) if grad_bias else None
    with torch.cuda.device(dev):
        n = lib().rlk_linear_logp_backward_workspace_size_for(_ptr(h2), N, H, ldh, _ptr(w2), V, ldw)
        if n == 0:
            raise RlkError(2, "rlk_linear_logp_backward_workspace_size_for")
        ws = torch.empty(n, dtype=torch.uint8, device=dev)
        dt = _DT[out_dtype]
        _check(lib().rlk_linear_logp_backward(
            _ptr(h2), N, H, ldh, _ptr(w2), V, ldw, _ptr(bias), _ptr(t1), tstride, _ptr(l1), _ptr(g1),
            _ptr(gh), dt, H, _ptr(gw), dt, H, _ptr(gb), _ptr(ws), n, _stream_ptr(stream)),
            "rlk_linear_logp_backward")
    out = (None if gh is None else gh.reshape(*lead, H), gw, gb)
    if return_grad_logits:
        ldG = -(-V // 8) * 8
        G = ws[:N * ldG * 2].view(torch.bfloat16).view(N, ldG)[:, :V]
        out = out + (G,)
    return out


class _LinearLogpGrad(torch.autograd.Function):
    """Autograd wiring of rlk_linear_logp (forward) and rlk_linear_logp_backward: the
    forward keeps lse, the backward asks the library for the gradients autograd
    needs (BF16 for hidden and weight, FP32 for the bias).  lse is returned as a
    constant: gradients flow through logp only."""

    @staticmethod
    def forward(ctx, hidden, weight, bias, target):
        with torch.no_grad():
            logp, lse = linear_logp(hidden.detach(), weight.detach(), target,
                                    None if bias is None else bias.detach())
        ctx.save_for_backward(hidden, weight, bias, target, lse)
        ctx.mark_non_differentiable(lse)
        return logp, lse

    @staticmethod
    def backward(ctx, grad_logp, _grad_lse):
        hidden, weight, bias, target, lse = ctx.saved_tensors
        want_h, want_w, want_b = ctx.needs_input_grad[:3]
        if grad_logp is None or not (want_h or want_w or want_b):
            return None, None, None, None
        gh, gw, gb = linear_logp_backward(hidden, weight, target, lse, grad_logp, bias,
                                          grad_hidden=want_h, grad_weight=want_w,
                                          grad_bias=bool(want_b and bias is not None))
        return gh, gw, gb, None


def linear_logp_trainable(hidden: torch.Tensor, weight: torch.Tensor, target: torch.Tensor,
                          bias: torch.Tensor | None = None):
    """logp, lse as linear_logp, differentiable through logp with respect to hidden,
    weight and bias (the fused backward: G = g * (onehot(target) - softmax(z)), then
    grad_hidden = G . W and grad_weight = G^T . hidden in fixed order).  lse carries
    no gradient.  linear_logp itself stays forward-only and rejects inputs that
    require grad."""
    return _LinearLogpGrad.apply(hidden, weight, bias, target)


# ------------------------------------------------------------------ det_gemm
def _gemm_ws(op, x, xdt, xld, y, ydt, yld, device):
    n = lib().rlk_det_gemm_workspace_size(op, _ptr(x), xdt, x.size(0), x.size(1), xld,
                                          _ptr(y), ydt, y.size(0), y.size(1), yld)
    return torch.empty(max(n, 1), dtype=torch.uint8, device=device), n


def _flatten_rows(t: torch.Tensor) -> torch.Tensor:
    return t.reshape(-1, t.size(-1)) if t.dim() != 2 else t


def det_gemm_fwd(A: torch.Tensor, B: torch.Tensor, out_dtype=torch.bfloat16, *, stream=None):
    """C = A . B; A [..., M, K] bf16 (leading dims flattened into rows), B [K, N] bf16."""
    _require_cuda(A, B)
    lead = A.shape[:-1]
    A2, lda = _matrix(_flatten_rows(A), "A")
    B2, ldb = _matrix(B, "B")
    M, K = A2.shape
    if B2.size(0) != K:
        raise ValueError("A and B disagree on K")
    N = B2.size(1)
    C = torch.empty(M, N, dtype=out_dtype, device=A.device)
    with torch.cuda.device(A.device):
        ws, n = _gemm_ws(RLK_GEMM_FWD, A2, RLK_BF16, lda, B2, RLK_BF16, ldb, A.device)
        _check(lib().rlk_det_gemm_fwd(_ptr(A2), M, K, lda, _ptr(B2), N, ldb, _ptr(C), _DT[out_dtype],
                                      N, _ptr(ws), n, _stream_ptr(stream)), "rlk_det_gemm_fwd")
    return C.reshape(*lead, N)


def det_gemm_da(dC: torch.Tensor, B: torch.Tensor, out_dtype=torch.bfloat16, *, stream=None):
    """dA = dC . B^T; dC [..., M, N] bf16 or fp32 (fp32 is rounded to bf16 first), B [K, N]."""
    _require_cuda(dC, B)
    lead = dC.shape[:-1]
    d2, lddc = _matrix(_flatten_rows(dC), "dC")
    B2, ldb = _matrix(B, "B")
    M, N = d2.shape
    K = B2.size(0)
    if B2.size(1) != N:
        raise ValueError("dC and B disagree on N")
    dA = torch.empty(M, K, dtype=out_dtype, device=dC.device)
    with torch.cuda.device(dC.device):
        ws, n = _gemm_ws(RLK_GEMM_DA, d2, _DT[d2.dtype], lddc, B2, RLK_BF16, ldb, dC.device)
        _check(lib().rlk_det_gemm_da(_ptr(d2), _DT[d2.dtype], M, N, lddc, _ptr(B2), K, ldb, _ptr(dA),
                                     _DT[out_dtype], K, _ptr(ws), n, _stream_ptr(stream)),
               "rlk_det_gemm_da")
    return dA.reshape(*lead, K)


def det_gemm_db(A: torch.Tensor, dC: torch.Tensor, out_dtype=torch.bfloat16, *, stream=None):
    """dB = A^T . dC summed over every row; A [..., M, K] bf16, dC [..., M, N] bf16 or fp32."""
    _require_cuda(A, dC)
    A2, lda = _matrix(_flatten_rows(A), "A")
    d2, lddc = _matrix(_flatten_rows(dC), "dC")
    M, K = A2.shape
    if d2.size(0) != M:
        raise ValueError("A and dC disagree on M")
    N = d2.size(1)
    dB = torch.empty(K, N, dtype=out_dtype, device=A.device)
    with torch.cuda.device(A.device):
        ws, n = _gemm_ws(RLK_GEMM_DB, A2, RLK_BF16, lda, d2, _DT[d2.dtype], lddc, A.device)
        _check(lib().rlk_det_gemm_db(_ptr(A2), M, K, lda, _ptr(d2), _DT[d2.dtype], N, lddc, _ptr(dB),
                                     _DT[out_dtype], N, _ptr(ws), n, _stream_ptr(stream)),
               "rlk_det_gemm_db")
    return dB


def det_gemm_fwd_accum_fp32_(C: torch.Tensor, A: torch.Tensor, B: torch.Tensor, *, stream=None):
    """In place: C (fp32 [M, N]) += A . B, the product formed as by det_gemm_fwd and
    added to C once, after the full K reduction."""
    _require_cuda(C, A, B)
    if C.dtype != torch.float32:
        raise TypeError("C must be float32")
    A2, lda = _matrix(A, "A")
    B2, ldb = _matrix(B, "B")
    if C.dim() != 2 or C.stride(1) != 1:
        raise ValueError("C must be a 2-D row-major tensor (it is updated in place)")
    M, K = A2.shape
    N = B2.size(1)
    if B2.size(0) != K or tuple(C.shape) != (M, N):
        raise ValueError("shape mismatch")
    ldc = C.stride(0) if M > 1 else N
    with torch.cuda.device(A.device):
        ws, n = _gemm_ws(RLK_GEMM_FWD_ACCUM, A2, RLK_BF16, lda, B2, RLK_BF16, ldb, A.device)
        _check(lib().rlk_det_gemm_fwd_accum_fp32(_ptr(A2), M, K, lda, _ptr(B2), N, ldb, _ptr(C), ldc,
                                                 _ptr(ws), n, _stream_ptr(stream)),
               "rlk_det_gemm_fwd_accum_fp32")
    return C


def det_linear(X: torch.Tensor, W: torch.Tensor, out_dtype=torch.bfloat16, *, stream=None):
    """Y = X . W^T with the weight stored [N, K]; X [..., K] bf16 (leading dims are rows)."""
    _require_cuda(X, W)
    lead = X.shape[:-1]
    X2, ldx = _matrix(_flatten_rows(X), "X")
    W2, ldw = _matrix(W, "W")
    M, K = X2.shape
    N = W2.size(0)
    if W2.size(1) != K:
        raise ValueError("W must be [N, K]")
    Y = torch.empty(M, N, dtype=out_dtype, device=X.device)
    with torch.cuda.device(X.device):
        ws, n = _gemm_ws(RLK_GEMM_LINEAR_FWD, X2, RLK_BF16, ldx, W2, RLK_BF16, ldw, X.device)
        _check(lib().rlk_det_linear_fwd(_ptr(X2), M, K, ldx, _ptr(W2), N, ldw, _ptr(Y), _DT[out_dtype],
                                        N, _ptr(ws), n, _stream_ptr(stream)), "rlk_det_linear_fwd")
    return Y.reshape(*lead, N)


def det_linear_dx(dY: torch.Tensor, W: torch.Tensor, out_dtype=torch.bfloat16, *, stream=None):
    """dX = dY . W for Y = X . W^T; dY [..., N] bf16 or fp32 (fp32 rounded to bf16 first)."""
    _require_cuda(dY, W)
    lead = dY.shape[:-1]
    d2, lddy = _matrix(_flatten_rows(dY), "dY")
    W2, ldw = _matrix(W, "W")
    M, N = d2.shape
    K = W2.size(1)
    if W2.size(0) != N:
        raise ValueError("W must be [N, K]")
    dX = torch.empty(M, K, dtype=out_dtype, device=dY.device)
    with torch.cuda.device(dY.device):
        ws, n = _gemm_ws(RLK_GEMM_LINEAR_DX, d2, _DT[d2.dtype], lddy, W2, RLK_BF16, ldw, dY.device)
        _check(lib().rlk_det_linear_dx(_ptr(d2), _DT[d2.dtype], M, N, lddy, _ptr(W2), K, ldw, _ptr(dX),
                                       _DT[out_dtype], K, _ptr(ws), n, _stream_ptr(stream)),
               "rlk_det_linear_dx")
    return dX.reshape(*lead, K)


def det_linear_dw(dY: torch.Tensor, X: torch.Tensor, out_dtype=torch.bfloat16, *, stream=None):
    """dW [N, K] = dY^T . X summed over every row; dY [..., N] bf16 or fp32, X [..., K] bf16."""
    _require_cuda(dY, X)
    d2, lddy = _matrix(_flatten_rows(dY), "dY")
    X2, ldx = _matrix(_flatten_rows(X), "X")
    M, N = d2.shape
    if X2.size(0) != M:
        raise ValueError("dY and X disagree on the row count")
    K = X2.size(1)
    dW = torch.empty(N, K, dtype=out_dtype, device=dY.device)
    with torch.cuda.device(dY.device):
        ws, n = _gemm_ws(RLK_GEMM_LINEAR_DW, d2, _DT[d2.dtype], lddy, X2, RLK_BF16, ldx, dY.device)
        _check(lib().rlk_det_linear_dw(_ptr(d2), _DT[d2.dtype], M, N, lddy, _ptr(X2), K, ldx, _ptr(dW),
                                       _DT[out_dtype], K, _ptr(ws), n, _stream_ptr(stream)),
               "rlk_det_linear_dw")
    return dW


def _two_grads(fn, size_fn, g, x, w, out_shapes, out_dtype, want, stream):
    g2, ldg = _matrix(_flatten_rows(g), "grad")
    x2, ldx = _matrix(_flatten_rows(x), "x")
    w2, ldw = _matrix(w, "w")
    M, N = g2.shape
    K = x2.size(1)
    dev = g.device
    outs = [torch.empty(*shp, dtype=out_dtype, device=dev) if want[i] else None
            for i, shp in enumerate(out_shapes(M, N, K))]
    gdt = _DT[g2.dtype]
    with torch.cuda.device(dev):
        n = size_fn(_ptr(g2), gdt, M, N, ldg, _ptr(x2), K, ldx, _ptr(w2), ldw)
        ws = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)
        dt = _DT[out_dtype]
        lds = [o.size(1) if o is not None else 1 for o in outs]
        _check(fn(_ptr(g2), gdt, M, N, ldg, _ptr(x2), K, ldx, _ptr(w2), ldw, _ptr(outs[0]), dt,
                  lds[0], _ptr(outs[1]), dt, lds[1], _ptr(ws), n, _stream_ptr(stream)),
               fn.__name__)
    return tuple(outs)


def det_gemm_backward(dC: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
                      out_dtype=torch.bfloat16, *, grad_a: bool = True, grad_b: bool = True,
                      stream=None):
    """(dA = dC . B^T, dB = A^T . dC) for C = A . B, from one dC (bf16 or fp32; an fp32
    dC is rounded to bf16 once and shared by both products).  Bitwise equal to
    det_gemm_da and det_gemm_db."""
    _require_cuda(dC, A, B)
    lib_ = lib()
    return _two_grads(lib_.rlk_det_gemm_backward, lib_.rlk_det_gemm_backward_workspace_size, dC, A,
                      B, lambda M, N, K: ((M, K), (K, N)), out_dtype, (grad_a, grad_b),
                      stream)


def det_linear_backward(dY: torch.Tensor, X: torch.Tensor, W: torch.Tensor,
                        out_dtype=torch.bfloat16, *, grad_x: bool = True, grad_w: bool = True,
                        stream=None):
    """(dX = dY . W, dW = dY^T . X) for Y = X . W^T with W [N, K], from one dY (an fp32 dY
    is rounded to bf16 once).  Bitwise equal to det_linear_dx and det_linear_dw."""
    _require_cuda(dY, X, W)
    lib_ = lib()
    return _two_grads(lib_.rlk_det_linear_backward, lib_.rlk_det_linear_backward_workspace_size, dY,
                      X, W, lambda M, N, K: ((M, K), (N, K)), out_dtype, (grad_x, grad_w),
                      stream)


# ------------------------------------------------------------------ autograd wiring
class _DetGemmGrad(torch.autograd.Function):
    """C = A . B under autograd: det_gemm_fwd forward; det_gemm_backward for the
    gradients autograd needs (an FP32 dC, from an FP32-output forward, is rounded
    to BF16 once before both products)."""

    @staticmethod
    def forward(ctx, A, B, out_dtype):
        with torch.no_grad():
            C = det_gemm_fwd(A.detach(), B.detach(), out_dtype)
        ctx.save_for_backward(A, B)
        return C

    @staticmethod
    def backward(ctx, dC):
        A, B = ctx.saved_tensors
        want_a, want_b = ctx.needs_input_grad[:2]
        if not (want_a or want_b):
            return None, None, None
        dA, dB = det_gemm_backward(dC, A, B, grad_a=want_a, grad_b=want_b)
        return (None if dA is None else dA.reshape(A.shape)), dB, None


class _DetLinearGrad(torch.autograd.Function):
    """Y = X . W^T (W stored [N, K]) under autograd: det_linear forward,
    det_linear_backward for dX and dW."""

    @staticmethod
    def forward(ctx, X, W, out_dtype):
        with torch.no_grad():
            Y = det_linear(X.detach(), W.detach(), out_dtype)
        ctx.save_for_backward(X, W)
        return Y

    @staticmethod
    def backward(ctx, dY):
        X, W = ctx.saved_tensors
        want_x, want_w = ctx.needs_input_grad[:2]
        if not (want_x or want_w):
            return None, None, None
        dX, dW = det_linear_backward(dY, X, W, grad_x=want_x, grad_w=want_w)
        return (None if dX is None else dX.reshape(X.shape)), dW, None


def det_gemm_trainable(A: torch.Tensor, B: torch.Tensor, out_dtype=torch.bfloat16):
    """det_gemm_fwd(A, B) differentiable with respect to A and B (BF16 gradients from
    the fixed-order det_gemm backward products)."""
    return _DetGemmGrad.apply(A, B, out_dtype)


def det_linear_trainable(X: torch.Tensor, W: torch.Tensor, out_dtype=torch.bfloat16):
    """det_linear(X, W) differentiable with respect to X and W: a deterministic,
    batch-invariant stand-in for a bias-free nn.Linear forward and backward."""
    return _DetLinearGrad.apply(X, W, out_dtype)
