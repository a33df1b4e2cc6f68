"""CPU oracle for the small-M FP8 block-scaled linear layer (numpy front end).

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this package.  It shares no code with the CUDA
library in ``fp8_block_scaled_token_gb300``; the two meet only on the seeded
raw inputs.

What each function follows is stated in ``oracle.c``.  In brief:

* ``e4m3_decode_table`` / ``e4m3_encode`` -- the E4M3 format named on
  "Kernel-Level Optimisations for LLM Inference and Training", section
  "Quantisation kernels" (read as the "fn" variant: bias 7, max 448, NaN at
  0x7F/0xFF, round to nearest even, saturating).
* ``quant_act`` -- the run-time cast of the inputs to FP8 ("The profiler said
  the kernel ran zero times", section "What the trace showed"), one fp32 scale
  per token per 128 consecutive K.
* ``quant_weight`` -- one fp32 scale per 128x128 weight block ("A 23% faster
  GPU kernel, and a model that did not move", section "Why this shape is
  hard"; "The profiler said the kernel ran zero times", section "The output
  layer, which did run").
* ``gemm_fp8`` -- Y = dequant(Aq) . dequant(Wq)^T accumulated in fp64 per
  128-wide K block, with the error-bound reference sum |a||w|.
* ``gemm_bf16`` -- the 16-bit output-layer product of the same page, fp64.
* ``round_bf16`` -- one fp64 -> bf16 rounding, nearest-even.
* ``mx_quant`` / ``mx_gemm`` -- the microscaling (MX) variant of the layer:
  E4M3 elements with one power-of-two scale per 32 values along K, the
  conversion of the OCP microscaling specification (the pages only name the
  MX formats, "Kernel-Level Optimisations for LLM Inference and Training").
* ``greedy`` -- the greedy next-token choice the output layer feeds ("The
  profiler said the kernel ran zero times", section "The output layer, which
  did run"): per token, the column of the largest bf16 logit, lowest column on
  ties.

Every function here has at least one pin in ``tests/test_oracle_*.py``.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_u8p = ctypes.POINTER(ctypes.c_uint8)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int)
_int = ctypes.c_int


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def default_threads() -> int:
    if hasattr(os, "sched_getaffinity"):
        return max(1, len(os.sched_getaffinity(0)))
    return max(1, os.cpu_count() or 1)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


class Oracle:
    """One loaded copy of liboracle.so (the default build, or a test mutant)."""

    def __init__(self, path):
        L = ctypes.CDLL(path)
        L.oracle_e4m3_decode.restype = ctypes.c_double
        L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_decode_table.restype = None
        L.oracle_e4m3_decode_table.argtypes = [_f64p]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        L.oracle_round_bf16.restype = ctypes.c_uint16
        L.oracle_round_bf16.argtypes = [ctypes.c_double]
        L.oracle_f32_to_bf16.restype = ctypes.c_uint16
        L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        L.oracle_quant_act.restype = _int
        L.oracle_quant_act.argtypes = [_u16p, _int, _int, _int, _u8p, _f32p]
        L.oracle_quant_weight.restype = _int
        L.oracle_quant_weight.argtypes = [ctypes.c_void_p, _int, _int, _int, _u8p, _f32p]
        L.oracle_gemm_fp8.restype = _int
        L.oracle_gemm_fp8.argtypes = [_u8p, _f32p, _u8p, _f32p, _int, _int, _int,
                                      _i32p, _int, _f64p, _f64p, _int]
        L.oracle_gemm_bf16.restype = _int
        L.oracle_gemm_bf16.argtypes = [_u16p, _u16p, _int, _int, _int,
                                       _i32p, _int, _f64p, _f64p, _int]
        L.oracle_mx_quant.restype = _int
        L.oracle_mx_quant.argtypes = [ctypes.c_void_p, _int, _int, _int, _u8p, _u8p]
        L.oracle_mx_gemm.restype = _int
        L.oracle_mx_gemm.argtypes = [_u8p, _u8p, _u8p, _u8p, _int, _int, _int, _i32p, _int, _f64p, _f64p, _int]
        L.oracle_greedy.restype = _int
        L.oracle_greedy.argtypes = [_u16p, _int, _int, _int, _i32p, _f32p]
        self.lib = L
        self.path = path

    # -- E4M3 ---------------------------------------------------------------
    def e4m3_decode_table(self) -> np.ndarray:
        """float64[256]: the value of every E4M3 code (NaN for 0x7F, 0xFF)."""
        out = np.empty(256, dtype=np.float64)
        self.lib.oracle_e4m3_decode_table(_ptr(out, ctypes.c_double))
        return out

    def e4m3_encode(self, values) -> np.ndarray:
        """uint8 codes of float32 values (nearest, ties to even, saturating)."""
        v = np.asarray(values, dtype=np.float32)
        enc = self.lib.oracle_e4m3_encode
        flat = v.reshape(-1)
        out = np.fromiter((enc(float(x)) for x in flat), dtype=np.uint8, count=flat.size)
        return out.reshape(v.shape)

    # -- bf16 ---------------------------------------------------------------
    def round_bf16(self, values) -> np.ndarray:
        """uint16 bf16 bit patterns of float64 values, one nearest-even
        rounding."""
        v = np.asarray(values, dtype=np.float64)
        rnd = self.lib.oracle_round_bf16
        flat = v.reshape(-1)
        out = np.fromiter((rnd(float(x)) for x in flat), dtype=np.uint16, count=flat.size)
        return out.reshape(v.shape)

    def f32_to_bf16_bits(self, w) -> np.ndarray:
        """bf16 bit patterns of float32 values, nearest-even (the 16-bit copy
        of an fp32 weight matrix)."""
        w = np.ascontiguousarray(np.asarray(w, dtype=np.float32))
        return self.round_bf16(w.astype(np.float64))

    # -- quantisation ---------------------------------------------------------
    def quant_act(self, x_bf16_bits, K=None):
        """Per-token, per-128 quantisation of bf16 activations.

        x_bf16_bits: uint16 [M, ldx] (bf16 bit patterns).  The first ``K``
        columns of each row are quantised (all of them when K is None).
        Returns (xq uint8 [M, K], xs float32 [M, K/128]).
        """
        x = np.ascontiguousarray(np.asarray(x_bf16_bits, dtype=np.uint16))
        M, ldx = x.shape
        K = ldx if K is None else int(K)
        xq = np.empty((M, K), dtype=np.uint8)
        xs = np.empty((M, K // 128 if K % 128 == 0 else 0), dtype=np.float32)
        rc = self.lib.oracle_quant_act(_ptr(x, ctypes.c_uint16), M, K, ldx,
                                       _ptr(xq, ctypes.c_uint8), _ptr(xs, ctypes.c_float))
        if rc != 0:
            raise ValueError("oracle_quant_act: bad shape M=%d K=%d ldx=%d" % (M, K, ldx))
        return xq, xs

    def quant_weight(self, w):
        """128x128-block quantisation of a weight matrix.

        w: float32 [N, K], or uint16 [N, K] holding bf16 bit patterns.
        Returns (wq uint8 [N, K], ws float32 [ceil(N/128), K/128]).
        """
        w = np.ascontiguousarray(w)
        if w.dtype == np.float32:
            dtype = 0
        elif w.dtype == np.uint16:
            dtype = 1
        else:
            raise TypeError("weights must be float32 or bf16 bit patterns (uint16)")
        N, K = w.shape
        wq = np.empty((N, K), dtype=np.uint8)
        ws = np.empty(((N + 127) // 128, K // 128 if K % 128 == 0 else 0), dtype=np.float32)
        rc = self.lib.oracle_quant_weight(w.ctypes.data_as(ctypes.c_void_p), dtype, N, K,
                                          _ptr(wq, ctypes.c_uint8), _ptr(ws, ctypes.c_float))
        if rc != 0:
            raise ValueError("oracle_quant_weight: bad shape N=%d K=%d" % (N, K))
        return wq, ws

    # -- products -------------------------------------------------------------
    @staticmethod
    def _cols(cols, N):
        if cols is None:
            return None, N, None
        c = np.ascontiguousarray(np.asarray(cols, dtype=np.int32))
        return c, int(c.size), _ptr(c, ctypes.c_int)

    def gemm_fp8(self, aq, as_, wq, ws, cols=None, nthreads=None):
        """fp64 block-scaled product.

        aq uint8 [M,K], as_ float32 [M,K/128], wq uint8 [N,K], ws float32
        [ceil(N/128),K/128].  Returns (y float64 [M, ncols], bound float64
        [M, ncols]) for the output columns ``cols`` (all N when None).
        """
        aq = np.ascontiguousarray(aq, dtype=np.uint8)
        as_ = np.ascontiguousarray(as_, dtype=np.float32)
        wq = np.ascontiguousarray(wq, dtype=np.uint8)
        ws = np.ascontiguousarray(ws, dtype=np.float32)
        M, K = aq.shape
        N = wq.shape[0]
        if wq.shape[1] != K:
            raise ValueError("K mismatch")
        c, ncols, cptr = self._cols(cols, N)
        y = np.empty((M, ncols), dtype=np.float64)
        bound = np.empty((M, ncols), dtype=np.float64)
        rc = self.lib.oracle_gemm_fp8(_ptr(aq, ctypes.c_uint8), _ptr(as_, ctypes.c_float),
                                      _ptr(wq, ctypes.c_uint8), _ptr(ws, ctypes.c_float),
                                      M, N, K, cptr, ncols,
                                      _ptr(y, ctypes.c_double), _ptr(bound, ctypes.c_double),
                                      nthreads or default_threads())
        if rc != 0:
            raise ValueError("oracle_gemm_fp8: bad arguments")
        return y, bound

    def gemm_bf16(self, x_bits, w_bits, cols=None, nthreads=None):
        """fp64 product of bf16 operands (bit patterns, uint16): y = x . w^T."""
        x = np.ascontiguousarray(x_bits, dtype=np.uint16)
        w = np.ascontiguousarray(w_bits, dtype=np.uint16)
        M, K = x.shape
        N = w.shape[0]
        if w.shape[1] != K:
            raise ValueError("K mismatch")
        c, ncols, cptr = self._cols(cols, N)
        y = np.empty((M, ncols), dtype=np.float64)
        bound = np.empty((M, ncols), dtype=np.float64)
        rc = self.lib.oracle_gemm_bf16(_ptr(x, ctypes.c_uint16), _ptr(w, ctypes.c_uint16),
                                       M, N, K, cptr, ncols,
                                       _ptr(y, ctypes.c_double), _ptr(bound, ctypes.c_double),
                                       nthreads or default_threads())
        if rc != 0:
            raise ValueError("oracle_gemm_bf16: bad arguments")
        return y, bound

    def linear_fp8(self, x_bf16_bits, w, cols=None, nthreads=None):
        """The whole layer from raw inputs: quantise X per token per 128,
        quantise W per 128x128 block, form the fp64 product.  Returns a dict
        with every intermediate."""
        xq, xs = self.quant_act(x_bf16_bits)
        wq, ws = self.quant_weight(w)
        y, bound = self.gemm_fp8(xq, xs, wq, ws, cols=cols, nthreads=nthreads)
        return {"xq": xq, "xs": xs, "wq": wq, "ws": ws, "y": y, "bound": bound}


    # -- MX (microscaling) E4M3 -------------------------------------------------
    def mx_quant(self, x):
        """1x32 power-of-two block quantisation along K (the OCP microscaling
        conversion).  x: float32 [rows, K], or uint16 bf16 bit patterns.
        Returns (codes uint8 [rows, K], scale bytes uint8 [rows, K/32]; the
        scale of a block is 2^(byte - 127))."""
        x = np.ascontiguousarray(x)
        if x.dtype == np.float32:
            dtype = 0
        elif x.dtype == np.uint16:
            dtype = 1
        else:
            raise TypeError("x must be float32 or bf16 bit patterns (uint16)")
        rows, K = x.shape
        codes = np.empty((rows, K), dtype=np.uint8)
        sb = np.empty((rows, K // 32 if K % 32 == 0 else 0), dtype=np.uint8)
        rc = self.lib.oracle_mx_quant(x.ctypes.data_as(ctypes.c_void_p), dtype, rows, K,
                                      _ptr(codes, ctypes.c_uint8), _ptr(sb, ctypes.c_uint8))
        if rc != 0:
            raise ValueError("oracle_mx_quant: bad shape or non-finite input")
        return codes, sb

    def mx_gemm(self, aq, as_bytes, wq, ws_bytes, cols=None, nthreads=None):
        """fp64 product of two MX operands: aq [M,K] / as_bytes [M,K/32] and
        wq [N,K] / ws_bytes [N,K/32].  Returns (y, bound) [M, ncols]."""
        aq = np.ascontiguousarray(aq, dtype=np.uint8)
        asb = np.ascontiguousarray(as_bytes, dtype=np.uint8)
        wq = np.ascontiguousarray(wq, dtype=np.uint8)
        wsb = np.ascontiguousarray(ws_bytes, dtype=np.uint8)
        M, K = aq.shape
        N = wq.shape[0]
        if wq.shape[1] != K:
            raise ValueError("K mismatch")
        c, ncols, cptr = self._cols(cols, N)
        y = np.empty((M, ncols), dtype=np.float64)
        bound = np.empty((M, ncols), dtype=np.float64)
        rc = self.lib.oracle_mx_gemm(_ptr(aq, ctypes.c_uint8), _ptr(asb, ctypes.c_uint8),
                                     _ptr(wq, ctypes.c_uint8), _ptr(wsb, ctypes.c_uint8), M, N, K, cptr, ncols,
                                     _ptr(y, ctypes.c_double), _ptr(bound, ctypes.c_double),
                                     nthreads or default_threads())
        if rc != 0:
            raise ValueError("oracle_mx_gemm: bad arguments")
        return y, bound

    # -- greedy token choice ----------------------------------------------------
    def greedy(self, y_bf16_bits, N=None):
        """Per token row of bf16 logits (uint16 bit patterns [M, ldy]): the
        column of the largest value among the first N (all when None), lowest
        column on ties, +0 == -0.  Returns (token int32 [M], logit float32 [M],
        a zero logit reported as +0)."""
        y = np.ascontiguousarray(np.asarray(y_bf16_bits, dtype=np.uint16))
        M, ldy = y.shape
        N = ldy if N is None else int(N)
        token = np.empty(M, dtype=np.int32)
        logit = np.empty(M, dtype=np.float32)
        rc = self.lib.oracle_greedy(_ptr(y, ctypes.c_uint16), M, N, ldy, _ptr(token, ctypes.c_int),
                                    _ptr(logit, ctypes.c_float))
        if rc != 0:
            raise ValueError("oracle_greedy: bad shape or NaN logits")
        return token, logit


_default = None


def default() -> Oracle:
    """The oracle as built from oracle.c (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle(_build.build())
    return _default


def mutant(n: int) -> Oracle:
    """A copy of the oracle with deliberate mistake number ``n`` planted."""
    return Oracle(_build.build(mutant=n))


def __getattr__(name):
    # Module-level shortcuts: oracle.quant_act(...) == oracle.default().quant_act(...)
    if name in ("e4m3_decode_table", "e4m3_encode", "round_bf16", "f32_to_bf16_bits",
                "quant_act", "quant_weight", "gemm_fp8", "gemm_bf16", "linear_fp8", "greedy",
                "mx_quant", "mx_gemm"):
        return getattr(default(), name)
    raise AttributeError(name)
