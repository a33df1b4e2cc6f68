"""Small-M FP8 block-scaled linear layer for GB300 (sm_103a).

Thin Python binding over the C ABI of ``lib/libfp8bs.so`` (declared in
``include/fp8bs.h``).  This module only marshals arguments: torch tensors
provide device memory and the current CUDA stream; every step of the layer
runs in the library's CUDA kernels.  There is no fallback: if the library is
missing or a call fails, a RuntimeError says why.

Entry points (same names as the C ABI):

* ``fp8_quant_act(x)`` -> (xq, xs): per-token, per-128 E4M3 cast of bf16 X.
* ``fp8_quant_weight_blocks(w, tiled=False)`` -> (wq, ws): 128x128-block
  E4M3 weights, row-major or one contiguous 16 KB run per block.
* ``fp8_blockscaled_gemm(aq, as_, wq, ws)`` -> Y bf16 (M up to 512).
* ``fp8_blockscaled_gemm_fused(x, wq, ws)`` -> Y bf16 (cast fused in).
* ``fp8_blockscaled_gemm_fused_greedy(x, wq, ws)`` -> (token, logit, Y):
  the same plus the greedy next-token choice (M up to 64).
* ``bf16_pack_weights_tiled(w)``, ``bf16_gemm_ref(x, w)`` -> Y bf16 (the
  16-bit output-layer baseline).
* ``fp8_mx_quant_weights(w)``, ``fp8_mx_quant_act(x)``, ``fp8_mx_gemm(...)``:
  the native block-scaled (MX) variant, one UE8M0 scale per 32 K.
* ``fp8_blockscaled_gemm_workspace_size``, ``make_workspace``,
  ``workspace_status``, ``split_plan``, ``gemm_schedule``, ``fused_route``:
  workspace and schedule queries.
"""
import contextlib
import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "lib", "libfp8bs.so")
DEBUG_LIB_PATH = os.path.join(PKG, "lib", "libfp8bs_debug.so")

FLAG_OVERLAP_PREV = 1
FLAG_WEIGHTS_TILED = 2
FLAG_PROLOGUE_CAST = 4
F32, BF16 = 0, 1

_lib = None


class Fp8bsError(RuntimeError):
    def __init__(self, fn, code, text):
        super().__init__("%s failed: %s (status %d)" % (fn, text, code))
        self.code = code


_loaded = {}


def lib():
    """The active copy of the library: libfp8bs.so, or libfp8bs_debug.so
    inside ``with debug_library():``.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        _lib = _load(LIB_PATH)
    return _lib


@contextlib.contextmanager
def debug_library():
    """Route every call of this module to libfp8bs_debug.so (the FP8BS_DEBUG
    build, with device-side bounds checks) inside the ``with`` block."""
    global _lib
    prev = lib()
    _lib = _load(DEBUG_LIB_PATH)
    try:
        yield _lib
    finally:
        _lib = prev


def _load(path):
    if path in _loaded:
        return _loaded[path]
    if not os.path.exists(path):
        raise RuntimeError("%s is not built (expected at %s); run "
                           "`python -c \"import __graft_entry__ as g; g.build()\"`" % (os.path.basename(path), path))
    L = ctypes.CDLL(path)
    vp, i, u, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_size_t
    L.fp8bs_status_string.restype = ctypes.c_char_p
    L.fp8bs_status_string.argtypes = [i]
    sigs = {
        "fp8_quant_act": [vp, i, i, i, vp, vp, u, vp],
        "fp8_quant_weight_blocks": [vp, i, i, i, vp, vp, vp],
        "fp8_quant_weight_blocks_tiled": [vp, i, i, i, vp, vp, vp],
        "bf16_pack_weights_tiled": [vp, i, i, vp, vp],
        "fp8_blockscaled_gemm_workspace_size": [i, i, i, ctypes.POINTER(sz)],
        "fp8_blockscaled_gemm": [vp, vp, vp, vp, vp, i, i, i, vp, sz, u, vp],
        "fp8_blockscaled_gemm_fused": [vp, i, vp, vp, vp, i, i, i, vp, sz, u, vp],
        "fp8_blockscaled_gemm_fused_greedy": [vp, i, vp, vp, vp, i, i, i, vp, vp, vp, sz, u, vp],
        "bf16_gemm_ref_workspace_size": [i, i, i, ctypes.POINTER(sz)],
        "bf16_gemm_ref": [vp, vp, vp, i, i, i, vp, sz, u, vp],
        "fp8bs_workspace_status": [vp, i, ctypes.POINTER(i)],
        "fp8bs_split_plan": [i, i, i, i, i, ctypes.POINTER(i), ctypes.POINTER(ctypes.c_longlong),
                             ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(ctypes.c_longlong)],
        "fp8bs_gemm_schedule": [i, i, i, i, ctypes.POINTER(i), ctypes.POINTER(i), ctypes.POINTER(i),
                                ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(i)],
        "fp8bs_fused_route": [i, i, i, i, ctypes.c_uint, ctypes.POINTER(i)],
        "fp8bs_testhook_gemm_stall": [vp, vp, vp, vp, vp, i, i, i, vp, sz, i, ctypes.c_ulonglong, vp],
        "fp8bs_testhook_kernel_runs": [i, i, ctypes.POINTER(ctypes.c_ulonglong)],
        "fp8bs_testhook_gemm_fused_sms": [vp, i, vp, vp, vp, i, i, i, vp, sz, u, i, vp],
        "fp8bs_testhook_workspace_size_sms": [i, i, i, i, ctypes.POINTER(sz)],
        "fp8bs_testhook_debug_bad_tile": [vp, vp, vp, vp, vp, i, i, i, vp, sz, i, ctypes.c_ulonglong, vp],
        "fp8_blockscaled_gemm_fused_noalloc": [vp, i, vp, vp, vp, i, i, i, u, vp],
        "fp8_mx_quant_weights": [vp, i, i, i, vp, vp, vp],
        "fp8_mx_quant_act": [vp, i, i, i, vp, vp, u, vp],
        "fp8_mx_gemm_workspace_size": [i, i, i, ctypes.POINTER(sz)],
        "fp8_mx_gemm": [vp, vp, vp, vp, vp, i, i, i, vp, sz, u, vp],
    }
    for name, args in sigs.items():
        f = getattr(L, name)
        f.restype = i
        f.argtypes = args
    L.fp8bs_testhook_debug_build.restype = i
    L.fp8bs_testhook_debug_build.argtypes = []
    _loaded[path] = L
    return L


def status_string(code):
    return lib().fp8bs_status_string(int(code)).decode()


def _check(fn, code):
    if code != 0:
        raise Fp8bsError(fn, code, status_string(code))


# ---------------------------------------------------------------- helpers
def _torch():
    import torch
    return torch


# The helpers below run on every call: an eager decode pass makes hundreds of
# them per step, and their host time is on the critical path whenever the
# layers are short (measured: 17.3 us a fused call with the stream taken from
# torch.cuda.current_stream() and the device from t.device, 10.1 us as here,
# 4.8 us of it in the library).
def _stream():
    """The current CUDA stream of the current device, as an integer handle."""
    torch = _torch()
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return raw(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _ptr(t):
    """Device address of a tensor (the c_void_p arguments take integers)."""
    return t.data_ptr() if t is not None else None


def _need(t, dtype, name, ndim=2):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor (there is no CPU path)" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if t.dim() != ndim:
        raise ValueError("%s must be %d-D" % (name, ndim))


def _rows_contiguous(t, name):
    if t.stride(-1) != 1:
        raise ValueError("%s must have unit stride along K" % name)


# ---------------------------------------------------------------- entry points
def scales_shape(M, K):
    """Shape of the activation scales for M tokens: (M, K/128) token-major up
    to 16 tokens, (K/128, M) K-block-major above."""
    kg = max(K // 128, 0)
    return (M, kg) if M <= 16 else (kg, M)


def fp8_quant_act(x, xq=None, xs=None, flags=0):
    """bf16 X [M, K] (row stride may exceed K) -> (xq uint8 [M,K], xs fp32 of
    scales_shape(M, K))."""
    torch = _torch()
    _need(x, torch.bfloat16, "x")
    _rows_contiguous(x, "x")
    M, K = x.shape
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if xs is None:
        xs = torch.empty(scales_shape(M, K), dtype=torch.float32, device=x.device)
    _check("fp8_quant_act", lib().fp8_quant_act(_ptr(x), M, K, x.stride(0), _ptr(xq), _ptr(xs), flags, _stream()))
    return xq, xs


def fp8_quant_weight_blocks(w, wq=None, ws=None, tiled=False):
    """fp32 or bf16 W [N, K] -> (wq, ws fp32 [ceil(N/128), K/128]).

    wq is uint8 [N, K] row-major, or with ``tiled=True`` uint8
    [ceil(N/128) * K/128, 128, 128]: one contiguous 128x128 block per weight
    tile (rows past N zero), for the GEMMs' tiled-weight mode."""
    torch = _torch()
    if w.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("w must be float32 or bfloat16")
    _need(w, w.dtype, "w")
    if not w.is_contiguous():
        raise ValueError("w must be contiguous")
    N, K = w.shape
    if wq is None:
        shape = (((N + 127) // 128) * max(K // 128, 0), 128, 128) if tiled else (N, K)
        wq = torch.empty(shape, dtype=torch.uint8, device=w.device)
    if ws is None:
        ws = torch.empty(((N + 127) // 128, max(K // 128, 0)), dtype=torch.float32, device=w.device)
    wt = BF16 if w.dtype == torch.bfloat16 else F32
    fn = lib().fp8_quant_weight_blocks_tiled if tiled else lib().fp8_quant_weight_blocks
    _check("fp8_quant_weight_blocks", fn(_ptr(w), wt, N, K, _ptr(wq), _ptr(ws), _stream()))
    return wq, ws


def bf16_pack_weights_tiled(w, wt=None):
    """bf16 W [N, K] -> bf16 [ceil(N/128) * K/64, 128, 64], one contiguous
    128x64 tile per block (rows past N zero), for bf16_gemm_ref(tiled)."""
    torch = _torch()
    _need(w, torch.bfloat16, "w")
    if not w.is_contiguous():
        raise ValueError("w must be contiguous")
    N, K = w.shape
    if wt is None:
        wt = torch.empty((((N + 127) // 128) * max(K // 64, 0), 128, 64), dtype=torch.bfloat16, device=w.device)
    _check("bf16_pack_weights_tiled", lib().bf16_pack_weights_tiled(_ptr(w), N, K, _ptr(wt), _stream()))
    return wt


def _weight_dims(wq, K, n, what):
    """(N, flag) of a row-major [N,K] or tiled [tiles,128,*] weight operand."""
    if wq.dim() == 2:
        if wq.shape[1] != K:
            raise ValueError("operand shapes do not agree")
        return wq.shape[0], 0
    if wq.dim() == 3 and wq.shape[1] == 128:
        if n is None:
            raise ValueError("%s is tiled: pass n= (the number of weight rows)" % what)
        if wq.numel() != ((int(n) + 127) // 128) * 128 * K:
            raise ValueError("tiled %s does not hold ceil(n/128)*128*K elements" % what)
        return int(n), FLAG_WEIGHTS_TILED
    raise ValueError("%s must be [N, K] or tiled [tiles, 128, *]" % what)


def fp8_blockscaled_gemm_workspace_size(M, N, K):
    n = ctypes.c_size_t(0)
    _check("fp8_blockscaled_gemm_workspace_size", lib().fp8_blockscaled_gemm_workspace_size(M, N, K, ctypes.byref(n)))
    return n.value


def bf16_gemm_ref_workspace_size(M, N, K):
    n = ctypes.c_size_t(0)
    _check("bf16_gemm_ref_workspace_size", lib().bf16_gemm_ref_workspace_size(M, N, K, ctypes.byref(n)))
    return n.value


def make_workspace(nbytes, device=None):
    """A zero-filled, 256-byte aligned device workspace of ``nbytes``."""
    torch = _torch()
    return torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")


def fp8_blockscaled_gemm(aq, as_, wq, ws, y=None, workspace=None, flags=0, n=None):
    """Y[M,N] bf16 from pre-quantised operands (wq row-major, or tiled with
    n= the number of weight rows)."""
    torch = _torch()
    _need(aq, torch.uint8, "aq")
    _need(as_, torch.float32, "as_")
    _need(wq, torch.uint8, "wq", ndim=wq.dim() if wq.dim() in (2, 3) else 2)
    _need(ws, torch.float32, "ws")
    for t, nm in ((aq, "aq"), (as_, "as_"), (wq, "wq"), (ws, "ws")):
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % nm)
    M, K = aq.shape
    N, tf = _weight_dims(wq, K, n, "wq")
    flags |= tf
    if tuple(as_.shape) != scales_shape(M, K) or tuple(ws.shape) != ((N + 127) // 128, K // 128):
        raise ValueError("operand shapes do not agree")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=aq.device)
    if workspace is None:
        workspace = make_workspace(fp8_blockscaled_gemm_workspace_size(M, N, K), aq.device)
    _check("fp8_blockscaled_gemm",
           lib().fp8_blockscaled_gemm(_ptr(aq), _ptr(as_), _ptr(wq), _ptr(ws), _ptr(y), M, N, K,
                                      _ptr(workspace), workspace.numel(), flags, _stream()))
    return y


def fp8_blockscaled_gemm_fused(x, wq, ws, y=None, workspace=None, flags=0, n=None):
    """Y[M,N] bf16 from bf16 activations (row stride may exceed K); wq
    row-major, or tiled with n= the number of weight rows."""
    torch = _torch()
    _need(x, torch.bfloat16, "x")
    _rows_contiguous(x, "x")
    _need(wq, torch.uint8, "wq", ndim=wq.dim() if wq.dim() in (2, 3) else 2)
    _need(ws, torch.float32, "ws")
    M, K = x.shape
    N, tf = _weight_dims(wq, K, n, "wq")
    flags |= tf
    if tuple(ws.shape) != ((N + 127) // 128, K // 128):
        raise ValueError("operand shapes do not agree")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = make_workspace(fp8_blockscaled_gemm_workspace_size(M, N, K), x.device)
    _check("fp8_blockscaled_gemm_fused",
           lib().fp8_blockscaled_gemm_fused(_ptr(x), x.stride(0), _ptr(wq), _ptr(ws), _ptr(y), M, N, K,
                                            _ptr(workspace), workspace.numel(), flags, _stream()))
    return y


def fp8_blockscaled_gemm_fused_greedy(x, wq, ws, y=None, store_y=True, token=None, logit=None, workspace=None,
                                      flags=0, n=None):
    """The fused layer plus the greedy next-token choice per token row:
    returns (token int32 [M], logit fp32 [M], y bf16 [M,N] or None).  With
    ``store_y=False`` the logits are not written (y must then be None)."""
    torch = _torch()
    _need(x, torch.bfloat16, "x")
    _rows_contiguous(x, "x")
    _need(wq, torch.uint8, "wq", ndim=wq.dim() if wq.dim() in (2, 3) else 2)
    _need(ws, torch.float32, "ws")
    M, K = x.shape
    N, tf = _weight_dims(wq, K, n, "wq")
    flags |= tf
    if tuple(ws.shape) != ((N + 127) // 128, K // 128):
        raise ValueError("operand shapes do not agree")
    if not store_y and y is not None:
        raise ValueError("store_y=False takes no y")
    if store_y and y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    if token is None:
        token = torch.empty((M,), dtype=torch.int32, device=x.device)
    if logit is None:
        logit = torch.empty((M,), dtype=torch.float32, device=x.device)
    _need(token, torch.int32, "token", ndim=1)
    _need(logit, torch.float32, "logit", ndim=1)
    if token.numel() < M or logit.numel() < M:
        raise ValueError("token and logit need M entries")
    if workspace is None:
        workspace = make_workspace(fp8_blockscaled_gemm_workspace_size(M, N, K), x.device)
    _check("fp8_blockscaled_gemm_fused_greedy",
           lib().fp8_blockscaled_gemm_fused_greedy(_ptr(x), x.stride(0), _ptr(wq), _ptr(ws),
                                                   _ptr(y) if y is not None else None, M, N, K, _ptr(token),
                                                   _ptr(logit), _ptr(workspace), workspace.numel(), flags,
                                                   _stream()))
    return token, logit, y


def bf16_gemm_ref(x, w, y=None, workspace=None, flags=0, n=None):
    """Y[M,N] bf16 = X bf16 [M,K] . W bf16 [N,K]^T (fp32 accumulation); w
    row-major, or tiled (bf16_pack_weights_tiled) with n= the weight rows."""
    torch = _torch()
    _need(x, torch.bfloat16, "x")
    _need(w, torch.bfloat16, "w", ndim=w.dim() if w.dim() in (2, 3) else 2)
    if not (x.is_contiguous() and w.is_contiguous()):
        raise ValueError("x and w must be contiguous")
    M, K = x.shape
    N, tf = _weight_dims(w, K, n, "w")
    flags |= tf
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = make_workspace(bf16_gemm_ref_workspace_size(M, N, K), x.device)
    _check("bf16_gemm_ref",
           lib().bf16_gemm_ref(_ptr(x), _ptr(w), _ptr(y), M, N, K, _ptr(workspace), workspace.numel(),
                               flags, _stream()))
    return y


# ---------------------------------------------------------------- MX variant
def fp8_mx_quant_weights(w, wq=None, ws_atoms=None):
    """fp32 or bf16 W [N, K] -> (wq uint8 [ceil(N/128) * K/128, 128, 128]
    tiled codes, ws_atoms uint8 [ceil(N/128) * K/128, 512] scale atoms):
    one power-of-two (UE8M0) scale per 32 K per row (include/fp8bs.h)."""
    torch = _torch()
    if w.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("w must be float32 or bfloat16")
    _need(w, w.dtype, "w")
    if not w.is_contiguous():
        raise ValueError("w must be contiguous")
    N, K = w.shape
    tiles = ((N + 127) // 128) * max(K // 128, 0)
    if wq is None:
        wq = torch.empty((tiles, 128, 128), dtype=torch.uint8, device=w.device)
    if ws_atoms is None:
        ws_atoms = torch.empty((tiles, 512), dtype=torch.uint8, device=w.device)
    wt = BF16 if w.dtype == torch.bfloat16 else F32
    _check("fp8_mx_quant_weights", lib().fp8_mx_quant_weights(_ptr(w), wt, N, K, _ptr(wq), _ptr(ws_atoms), _stream()))
    return wq, ws_atoms


def fp8_mx_quant_act(x, xq=None, xs_atoms=None, flags=0):
    """bf16 X [M, K] (M <= 512; row stride may exceed K) -> (xq uint8 [M, K],
    xs_atoms uint8 [ceil(M/128) * K/128, 512]: atom (token tile, K block))."""
    torch = _torch()
    _need(x, torch.bfloat16, "x")
    _rows_contiguous(x, "x")
    M, K = x.shape
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if xs_atoms is None:
        xs_atoms = torch.empty((((M + 127) // 128) * max(K // 128, 0), 512), dtype=torch.uint8, device=x.device)
    _check("fp8_mx_quant_act", lib().fp8_mx_quant_act(_ptr(x), M, K, x.stride(0), _ptr(xq), _ptr(xs_atoms), flags,
                                                      _stream()))
    return xq, xs_atoms


def fp8_mx_gemm_workspace_size(M, N, K):
    n = ctypes.c_size_t(0)
    _check("fp8_mx_gemm_workspace_size", lib().fp8_mx_gemm_workspace_size(M, N, K, ctypes.byref(n)))
    return n.value


def fp8_mx_gemm(aq, as_atoms, wq, ws_atoms, n, y=None, workspace=None, flags=0):
    """Y[M, n] bf16 from MX operands (fp8_mx_quant_act / fp8_mx_quant_weights;
    n = the number of weight rows)."""
    torch = _torch()
    _need(aq, torch.uint8, "aq")
    _need(as_atoms, torch.uint8, "as_atoms")
    _need(wq, torch.uint8, "wq", ndim=3)
    _need(ws_atoms, torch.uint8, "ws_atoms")
    M, K = aq.shape
    N = int(n)
    tiles = ((N + 127) // 128) * (K // 128)
    if (wq.numel() != tiles * 16384 or ws_atoms.numel() != tiles * 512 or
            as_atoms.numel() != ((M + 127) // 128) * (K // 128) * 512):
        raise ValueError("operand shapes do not agree")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=aq.device)
    if workspace is None:
        workspace = make_workspace(fp8_mx_gemm_workspace_size(M, N, K), aq.device)
    _check("fp8_mx_gemm", lib().fp8_mx_gemm(_ptr(aq), _ptr(as_atoms), _ptr(wq), _ptr(ws_atoms), _ptr(y), M, N, K,
                                            _ptr(workspace), workspace.numel(), flags, _stream()))
    return y


def workspace_status(workspace, clear=False):
    """Device-side failure word of a workspace (synchronises the device)."""
    code = ctypes.c_int(0)
    rc = lib().fp8bs_workspace_status(_ptr(workspace), 1 if clear else 0, ctypes.byref(code))
    if rc not in (0, 7):
        _check("fp8bs_workspace_status", rc)
    return code.value


def split_plan(N, K, bf16=False, num_sms=0, cta=-1):
    """(ctas, units, unit_begin, unit_end) of the K-split schedule."""
    c = ctypes.c_int(0)
    u = ctypes.c_longlong(0)
    b = ctypes.c_longlong(0)
    e = ctypes.c_longlong(0)
    _check("fp8bs_split_plan", lib().fp8bs_split_plan(N, K, 1 if bf16 else 0, num_sms, cta, ctypes.byref(c),
                                                      ctypes.byref(u), ctypes.byref(b), ctypes.byref(e)))
    return c.value, u.value, (b.value if cta >= 0 else None), (e.value if cta >= 0 else None)


def fused_route(M, N, K, num_sms=0, flags=0):
    """'prologue' when fp8_blockscaled_gemm_fused casts the activations in the
    GEMM kernel's prologue for this shape and flags (FLAG_PROLOGUE_CAST, where
    the cache fits), 'separate' when it runs the cast as its own kernel first."""
    v = ctypes.c_int(0)
    _check("fp8bs_fused_route", lib().fp8bs_fused_route(M, N, K, num_sms, flags, ctypes.byref(v)))
    return "prologue" if v.value else "separate"


def gemm_schedule(M, N, K, num_sms=0):
    """dict(npad, token_tiles, ctas, units, split) the FP8 GEMMs use for M tokens."""
    v = [ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0), ctypes.c_longlong(0), ctypes.c_int(0)]
    _check("fp8bs_gemm_schedule", lib().fp8bs_gemm_schedule(M, N, K, num_sms, *[ctypes.byref(a) for a in v]))
    return dict(npad=v[0].value, token_tiles=v[1].value, ctas=v[2].value, units=v[3].value, split=bool(v[4].value))
