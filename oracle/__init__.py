"""FP64 CPU oracle — TEST INFRASTRUCTURE ONLY.

Only the test suite, the package smoke check and the benchmark's CPU-baseline
and reference legs may import this package.  The product path never does, and
this package never imports the product package: the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, double precision, no FMA
contraction, no fast-math).  This module compiles it with gcc on first use and
marshals numpy arrays through ctypes.

Definitions (web pages of the RL-Kernel project):
  * linear_logp — "feat(linear-logp): add batch-invariant fused SM90 operator",
    Walkthrough and PR body: logits = hidden . W^T (+ bias), log-sum-exp over
    the vocabulary, gather of the target logit; returns logp and lse.
  * gemm_fwd / gemm_da / gemm_db — "feat(musa): add native deterministic gemm
    kernel", Summary: C = A B, dA = dC B^T, dB = A^T dC; and its review
    comment: on an FP32-output backward, grad_output is rounded to BF16 first
    (``f32_to_bf16_rne``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
LIB_PATH = os.path.join(_HERE, "liboracle.so")

_CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-std=c11"]


def build(out_path: str = LIB_PATH, mutant: int = 0, openmp: bool = True) -> str:
    """Compile oracle.c into a shared library (``mutant`` > 0 plants a test mistake)."""
    cmd = ["gcc", *_CFLAGS]
    if openmp:
        cmd.append("-fopenmp")
    if mutant:
        cmd.append(f"-DORACLE_MUTANT={int(mutant)}")
    tmp = out_path + f".tmp{os.getpid()}"
    cmd += [_SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(cmd, check=True, capture_output=True, text=True)
    except subprocess.CalledProcessError as e:
        if openmp:  # a toolchain without libgomp still gets a (single-threaded) oracle
            return build(out_path, mutant, openmp=False)
        raise RuntimeError(f"oracle build failed: {e.stderr}") from e
    os.replace(tmp, out_path)
    return out_path


def _needs_build() -> bool:
    return (not os.path.exists(LIB_PATH)
            or os.path.getmtime(LIB_PATH) < os.path.getmtime(_SRC))


_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def _bind(lib):
    lib.oracle_linear_logp.argtypes = [_P, _I64, _I64, _I64, _P, _I64, _I64, _P, _P, _I64,
                                       _P, _I64, _P, _P, _P, ctypes.c_int]
    lib.oracle_linear_logp.restype = ctypes.c_int
    lib.oracle_linear_logp_grad_logits.argtypes = [_P, _I64, _I64, _I64, _P, _I64, _I64, _P, _P,
                                                   _I64, _P, _P, ctypes.c_int]
    lib.oracle_linear_logp_grad_logits.restype = ctypes.c_int
    lib.oracle_logits.argtypes = [_P, _I64, _I64, _I64, _P, _I64, _I64, _P, _P]
    lib.oracle_logits.restype = None
    for name in ("oracle_gemm_fwd", "oracle_gemm_da", "oracle_gemm_db"):
        f = getattr(lib, name)
        f.argtypes = [_P, _I64, _I64, _I64, _P, _I64, _I64, _P, _I64, _P, ctypes.c_int]
        f.restype = None
    lib.oracle_f32_to_bf16_rne_array.argtypes = [_P, _P, _I64]
    lib.oracle_f64_to_bf16_rne_array.argtypes = [_P, _P, _I64]
    lib.oracle_f32_to_bf16_rne.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16_rne.restype = ctypes.c_uint16
    lib.oracle_f64_to_bf16_rne.argtypes = [ctypes.c_double]
    lib.oracle_f64_to_bf16_rne.restype = ctypes.c_uint16
    lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f64.restype = ctypes.c_double
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


class Oracle:
    """ctypes front end of one compiled oracle library (the real one or a mutant)."""

    def __init__(self, path: str):
        self.path = path
        self.lib = _bind(ctypes.CDLL(path))

    # -- helpers ---------------------------------------------------------
    @staticmethod
    def _u16(a) -> np.ndarray:
        a = np.ascontiguousarray(a)
        if a.dtype != np.uint16:
            raise TypeError("BF16 operands are passed as uint16 bit patterns")
        return a

    @staticmethod
    def _ptr(a):
        return None if a is None else a.ctypes.data_as(ctypes.c_void_p)

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    # -- conversions -----------------------------------------------------
    def bf16_to_f64(self, bits) -> np.ndarray:
        bits = self._u16(bits)
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)

    def f32_to_bf16_rne(self, x) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.float32)
        out = np.empty(x.shape, dtype=np.uint16)
        self.lib.oracle_f32_to_bf16_rne_array(self._ptr(x), self._ptr(out), x.size)
        return out

    def f64_to_bf16_rne(self, x) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.float64)
        out = np.empty(x.shape, dtype=np.uint16)
        self.lib.oracle_f64_to_bf16_rne_array(self._ptr(x), self._ptr(out), x.size)
        return out

    # -- linear log-probability -------------------------------------------
    def logits(self, hidden, weight, bias=None) -> np.ndarray:
        hidden, weight = self._u16(hidden), self._u16(weight)
        N, H = hidden.shape
        V = weight.shape[0]
        b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
        z = np.empty((N, V), dtype=np.float64)
        self.lib.oracle_logits(self._ptr(hidden), N, H, H, self._ptr(weight), V, H,
                               self._ptr(b), self._ptr(z))
        return z

    def linear_logp(self, hidden, weight, target, bias=None, rows=None, threads: int = 0,
                    target_stride: int = 1):
        """Returns (logp, lse, z_target) as float64 arrays over ``rows`` (default: all)."""
        hidden, weight = self._u16(hidden), self._u16(weight)
        N, H = hidden.shape
        V, Hw = weight.shape
        if Hw != H:
            raise ValueError("hidden and weight disagree on H")
        target = np.ascontiguousarray(target, dtype=np.int64)
        b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
        r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        count = N if r is None else r.size
        logp = np.empty(count, np.float64)
        lse = np.empty(count, np.float64)
        zt = np.empty(count, np.float64)
        rc = self.lib.oracle_linear_logp(self._ptr(hidden), N, H, H, self._ptr(weight), V, H,
                                         self._ptr(b), self._ptr(target), target_stride,
                                         self._ptr(r), count, self._ptr(logp), self._ptr(lse),
                                         self._ptr(zt), threads)
        if rc != 0:
            raise MemoryError("oracle scratch allocation failed")
        return logp, lse, zt

    # -- backward of linear log-probability --------------------------------
    def grad_logits(self, hidden, weight, target, grad, bias=None, threads: int = 0,
                    target_stride: int = 1) -> np.ndarray:
        """G = dL/dz [N, V] for L = sum_r grad[r] * logp[r] (small cases)."""
        hidden, weight = self._u16(hidden), self._u16(weight)
        N, H = hidden.shape
        V = weight.shape[0]
        target = np.ascontiguousarray(target, dtype=np.int64)
        g = np.ascontiguousarray(grad, dtype=np.float64)
        b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
        G = np.empty((N, V), np.float64)
        rc = self.lib.oracle_linear_logp_grad_logits(
            self._ptr(hidden), N, H, H, self._ptr(weight), V, H, self._ptr(b), self._ptr(target),
            target_stride, self._ptr(g), self._ptr(G), threads)
        if rc != 0:
            raise MemoryError("oracle scratch allocation failed")
        return G

    def linear_logp_backward(self, hidden, weight, target, grad, bias=None, threads: int = 0):
        """(grad_hidden [N,H], grad_weight [V,H], grad_bias [V], G [N,V]) in float64.

        G from grad_logits (the definition); the three reductions of G are library
        float64 matrix products / sums (numpy) over the decoded BF16 inputs."""
        G = self.grad_logits(hidden, weight, target, grad, bias, threads)
        hd = self.bf16_to_f64(hidden)
        wd = self.bf16_to_f64(weight)
        return G @ wd, G.T @ hd, G.sum(axis=0), G

    # -- deterministic GEMM family ----------------------------------------
    def gemm_fwd(self, A, B, rows=None, threads: int = 0) -> np.ndarray:
        A, B = self._u16(A), self._u16(B)
        M, K = A.shape
        K2, N = B.shape
        assert K2 == K
        r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        count = M if r is None else r.size
        C = np.empty((count, N), np.float64)
        self.lib.oracle_gemm_fwd(self._ptr(A), M, K, K, self._ptr(B), N, N,
                                 self._ptr(r), count, self._ptr(C), threads)
        return C

    def gemm_da(self, dC, B, rows=None, threads: int = 0) -> np.ndarray:
        dC, B = self._u16(dC), self._u16(B)
        M, N = dC.shape
        K, N2 = B.shape
        assert N2 == N
        r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        count = M if r is None else r.size
        dA = np.empty((count, K), np.float64)
        self.lib.oracle_gemm_da(self._ptr(dC), M, N, N, self._ptr(B), K, N,
                                self._ptr(r), count, self._ptr(dA), threads)
        return dA

    def gemm_db(self, A, dC, rows=None, threads: int = 0) -> np.ndarray:
        A, dC = self._u16(A), self._u16(dC)
        M, K = A.shape
        M2, N = dC.shape
        assert M2 == M
        r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        count = K if r is None else r.size
        dB = np.empty((count, N), np.float64)
        self.lib.oracle_gemm_db(self._ptr(A), M, K, K, self._ptr(dC), N, N,
                                self._ptr(r), count, self._ptr(dB), threads)
        return dB


_ORACLE = None


def load() -> Oracle:
    """The real oracle, compiled on first use."""
    global _ORACLE
    if _ORACLE is None:
        if _needs_build():
            build()
        _ORACLE = Oracle(LIB_PATH)
    return _ORACLE


def load_mutant(mutant: int) -> Oracle:
    """An oracle with a planted mistake (see ORACLE_MUTANT in oracle.c)."""
    d = tempfile.mkdtemp(prefix="oracle_mutant_")
    return Oracle(build(os.path.join(d, f"liboracle_m{mutant}.so"), mutant=mutant))
