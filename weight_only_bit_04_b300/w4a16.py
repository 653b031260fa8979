"""Python binding of libw4a16.so (ctypes).

Argument marshalling only: tensors are checked, their device pointers and the
current CUDA stream are passed to the C ABI declared in include/w4a16.h, and a
non-OK status becomes a ``W4A16Error``. Every step of the computation runs in
the library's CUDA kernels; PyTorch provides device memory and streams.
If the shared library is missing this module raises on first use -- there is
no fallback.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libw4a16.so")

STATUS = {
    0: "W4A16_OK",
    1: "W4A16_ERR_INVALID_ARG",
    2: "W4A16_ERR_UNSUPPORTED",
    3: "W4A16_ERR_MISALIGNED",
    4: "W4A16_ERR_BUFFER_TOO_SMALL",
    5: "W4A16_ERR_CUDA",
}

# Exported entry points (name -> (restype, argtypes)).
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t


class Format(ctypes.Structure):
    """Mirror of ``w4a16_format``."""

    _fields_ = [
        ("bits", ctypes.c_int32),
        ("group_size", ctypes.c_int32),
        ("symmetric", ctypes.c_int32),
        ("has_g_idx", ctypes.c_int32),
        ("N", ctypes.c_int64),
        ("K", ctypes.c_int64),
        ("has_act_scale", ctypes.c_int32),
    ]

    def __repr__(self):
        return (f"Format(bits={self.bits}, group_size={self.group_size}, symmetric={self.symmetric}, "
                f"has_g_idx={self.has_g_idx}, N={self.N}, K={self.K}, has_act_scale={self.has_act_scale})")

    @property
    def G(self) -> int:
        return self.K // self.group_size


_FP = ctypes.POINTER(Format)


class ChainLayer(ctypes.Structure):
    """Mirror of ``w4a16_chain_layer``."""

    _fields_ = [
        ("packed", ctypes.c_void_p),
        ("packed_bytes", ctypes.c_size_t),
        ("x", ctypes.c_void_p),
        ("y", ctypes.c_void_p),
        ("wait_lo", ctypes.c_int32),
        ("wait_hi", ctypes.c_int32),
    ]


class ChainInfo(ctypes.Structure):
    """Mirror of ``w4a16_chain_info``."""

    _fields_ = [
        ("n_layers", ctypes.c_int32),
        ("bits", ctypes.c_int32),
        ("group_size", ctypes.c_int32),
        ("symmetric", ctypes.c_int32),
        ("M", ctypes.c_int64),
        ("n_slices", ctypes.c_int64),
        ("blocks", ctypes.c_int32),
        ("flags", ctypes.c_int32),
        ("reserved_x", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]

SIGNATURES = {
    "w4a16_packed_bytes": (_SZ, [_FP]),
    "w4a16_check_format": (ctypes.c_int, [_FP]),
    "w4a16_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "w4a16_last_cuda_error": (ctypes.c_int, []),
    "w4a16_quantize_workspace_bytes": (_SZ, [_FP]),
    "w4a16_quantize_rtn": (ctypes.c_int, [_FP, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "w4a16_quantize_rtn_noalloc": (ctypes.c_int, [_FP, _P, _P, _P, _P, _P, _P]),
    "w4a16_pack": (ctypes.c_int, [_FP, _P, _P, _P, _P, _P, _SZ, _P]),
    "w4a16_quantize_rtn_awq": (ctypes.c_int, [_FP, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "w4a16_pack_awq": (ctypes.c_int, [_FP, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "w4a16_dequant": (ctypes.c_int, [_FP, _P, _SZ, _P, _P]),
    "w4a16_gemv": (ctypes.c_int, [_FP, _P, _SZ, _P, _P, _I64, _P]),
    "w4a16_gemv_ex": (ctypes.c_int, [_FP, _P, _SZ, _P, _P, _I64, _I32, _I32, ctypes.c_uint32, _P]),
    "w4a16_gemm_workspace_bytes": (_SZ, [_FP, _I64]),
    "w4a16_gemm": (ctypes.c_int, [_FP, _P, _SZ, _P, _P, _I64, _P, _SZ, _P]),
    "w4a16_gemm_ex": (ctypes.c_int, [_FP, _P, _SZ, _P, _P, _I64, _P, _SZ, _I32, _I32, _P]),
    "w4a16_pipeline_timeouts": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32)]),
    "w4a16_set_wait_limit_ns": (ctypes.c_uint64, [ctypes.c_uint64]),
    "w4a16_debug_fail_next_launch": (None, [ctypes.c_int]),
    "w4a16_debug_check_word": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32)]),
    "w4a16_chain_workspace_bytes": (_SZ, [_FP, _I32, _I64]),
    "w4a16_gptq_workspace_bytes": (_SZ, [_FP]),
    "w4a16_gemv_grouped": (ctypes.c_int, [_FP, ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_size_t),
                                          _I32, _P, ctypes.POINTER(ctypes.c_void_p), _I64, ctypes.c_uint32, _P]),
    "w4a16_gptq": (ctypes.c_int, [_FP, _P, _P, _I64, ctypes.c_double, _P, _P, _P, _P, _P, _SZ, _P]),
    "w4a16_chain_prepare": (ctypes.c_int, [_FP, ctypes.POINTER(ChainLayer), _I32, _I64, _P, _SZ,
                                           ctypes.POINTER(ChainInfo)]),
    "w4a16_chain_run": (ctypes.c_int, [ctypes.POINTER(ChainInfo), _P, _P]),
}

_lib = None
_lock = threading.Lock()


class W4A16Error(RuntimeError):
    def __init__(self, fn: str, status: int, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        msg = f"{fn} returned {STATUS.get(status, status)}"
        if status == 5:
            msg += f" (cudaError {cuda_error})"
        super().__init__(msg)


def lib() -> ctypes.CDLL:
    """Load libw4a16.so (once). Raises if it has not been built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it with `python -m weight_only_bit_04_b300.build`")
                handle = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = handle
    return _lib


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise W4A16Error(fn, status, lib().w4a16_last_cuda_error() if status == 5 else 0)


def make_format(N: int, K: int, group_size: int = 128, symmetric: bool = False,
                has_g_idx: bool = False, bits: int = 4, act_scale: bool = False) -> Format:
    """``act_scale``: the layer carries an unfolded AWQ per-input-channel scale."""
    return Format(bits, group_size, int(bool(symmetric)), int(bool(has_g_idx)), N, K, int(bool(act_scale)))


def packed_bytes(fmt: Format) -> int:
    return int(lib().w4a16_packed_bytes(ctypes.byref(fmt)))


def check_format(fmt: Format) -> int:
    return int(lib().w4a16_check_format(ctypes.byref(fmt)))


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        if stream.device.index != torch.cuda.current_device():
            raise ValueError(f"stream is on {stream.device}, the current device is cuda:{torch.cuda.current_device()}")
        return stream.cuda_stream
    return int(stream)


def _keep_alive(stream, *tensors) -> None:
    """Tensors allocated here and used by a kernel on a caller-given stream:
    tell the caching allocator, so that their memory is not handed out again
    before that stream's work is done."""
    if stream is None:
        return
    s = stream if isinstance(stream, torch.cuda.Stream) else torch.cuda.ExternalStream(int(stream))
    for t in tensors:
        if t is not None:
            t.record_stream(s)


def _dev(t: torch.Tensor, dtype: torch.dtype, name: str, shape=None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, the current device is cuda:{torch.cuda.current_device()}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def _host_gidx(g_idx, K: int):
    if g_idx is None:
        return None, None
    arr = torch.as_tensor(g_idx).to(device="cpu", dtype=torch.int32).contiguous()
    if arr.shape != (K,):
        raise ValueError("g_idx must have shape [K]")
    return arr, arr.data_ptr()


def quantize_rtn(fmt: Format, w: torch.Tensor, g_idx=None, act_scale=None, stream=None):
    """Round-to-nearest group quantization on the GPU -> (q uint8, scales fp16, zeros uint8|None).

    With ``fmt.has_act_scale`` pass ``act_scale`` (fp16 [K]): the quantized
    weights are fp16(w * act_scale) (unfolded AWQ).
    """
    N, K, G = fmt.N, fmt.K, fmt.G
    dev = w.device
    wp = _dev(w, torch.float16, "w", (N, K))
    ap = None if act_scale is None else _dev(act_scale, torch.float16, "act_scale", (K,))
    q = torch.empty((N, K), dtype=torch.uint8, device=dev)
    scales = torch.empty((N, G), dtype=torch.float16, device=dev)
    zeros = None if fmt.symmetric else torch.empty((N, G), dtype=torch.uint8, device=dev)
    ws_bytes = int(lib().w4a16_quantize_workspace_bytes(ctypes.byref(fmt)))
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    gi, gip = _host_gidx(g_idx, K)
    zp = None if zeros is None else zeros.data_ptr()
    wsp = ws.data_ptr() if ws_bytes else None
    if fmt.has_act_scale:
        st = lib().w4a16_quantize_rtn_awq(ctypes.byref(fmt), wp, ap, gip, q.data_ptr(), scales.data_ptr(), zp,
                                          wsp, ws_bytes, _stream(stream))
        _check("w4a16_quantize_rtn_awq", st)
    else:
        if ap is not None:
            raise ValueError("act_scale given but the format has no act scale")
        st = lib().w4a16_quantize_rtn(ctypes.byref(fmt), wp, gip, q.data_ptr(), scales.data_ptr(), zp,
                                      wsp, ws_bytes, _stream(stream))
        _check("w4a16_quantize_rtn", st)
    _keep_alive(stream, ws, q, scales, zeros)
    return q, scales, zeros


def gemv_grouped(fmts, packeds, x: torch.Tensor, outs=None, weights_ready: bool = False,
                 inputs_ready: bool = False, register_ring: bool = False, async_copy: bool = False, stream=None):
    """y_m = x . W_hat_m^T for up to 4 layers sharing x, K and the format, in one launch."""
    n = len(fmts)
    M = x.shape[0]
    K = fmts[0].K
    xp = _dev(x, torch.float16, "x", (M, K))
    allocated = outs is None
    if allocated:
        outs = [torch.empty((M, f.N), dtype=torch.float16, device=x.device) for f in fmts]
    fa = (Format * n)(*fmts)
    pa = (ctypes.c_void_p * n)(*[_dev(p, torch.uint8, "packed") for p in packeds])
    ba = (ctypes.c_size_t * n)(*[p.numel() for p in packeds])
    ya = (ctypes.c_void_p * n)(*[_dev(y, torch.float16, "out", (M, f.N)) for y, f in zip(outs, fmts)])
    flags = ((GEMV_WEIGHTS_READY if weights_ready else 0) | (GEMV_INPUTS_READY if inputs_ready else 0) |
             (GEMV_REGISTER_RING if register_ring else 0) | (GEMV_ASYNC_COPY if async_copy else 0))
    st = lib().w4a16_gemv_grouped(fa, pa, ba, n, xp, ya, M, flags, _stream(stream))
    _check("w4a16_gemv_grouped", st)
    if allocated:
        _keep_alive(stream, *outs)
    return outs


def gptq(fmt: Format, w: torch.Tensor, x: torch.Tensor, damp: float = 0.01, stream=None):
    """GPTQ on the GPU -> (q uint8, scales fp16, zeros uint8|None, g_idx host int32 ndarray|None).

    ``x``: fp16 [T, K] calibration activations. With ``fmt.has_g_idx`` the
    columns are taken by descending diag(H) and the act-order map is returned
    (on the host, ready for ``pack``).
    """
    N, K, G = fmt.N, fmt.K, fmt.G
    dev = w.device
    wp = _dev(w, torch.float16, "w", (N, K))
    if x.dim() != 2 or x.shape[1] != K:
        raise ValueError("x must be [T, K]")
    xp = _dev(x, torch.float16, "x", (x.shape[0], K))
    q = torch.empty((N, K), dtype=torch.uint8, device=dev)
    scales = torch.empty((N, G), dtype=torch.float16, device=dev)
    zeros = None if fmt.symmetric else torch.empty((N, G), dtype=torch.uint8, device=dev)
    gidx = torch.empty(K, dtype=torch.int32, device=dev) if fmt.has_g_idx else None
    nbytes = int(lib().w4a16_gptq_workspace_bytes(ctypes.byref(fmt)))
    if nbytes == 0:
        _check("w4a16_gptq", check_format(fmt) or 2)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    st = lib().w4a16_gptq(ctypes.byref(fmt), wp, xp, x.shape[0], float(damp), q.data_ptr(), scales.data_ptr(),
                          None if zeros is None else zeros.data_ptr(), None if gidx is None else gidx.data_ptr(),
                          ws.data_ptr(), nbytes, _stream(stream))
    _check("w4a16_gptq", st)
    _keep_alive(stream, ws, q, scales, zeros, gidx)
    return q, scales, zeros, (None if gidx is None else gidx.cpu().numpy())


def pack(fmt: Format, q: torch.Tensor, scales: torch.Tensor, zeros=None, g_idx=None,
         out: torch.Tensor | None = None, stream=None, act_scale=None) -> torch.Tensor:
    """Pack canonical codes/scales/zeros (and the act scale, fp16 [K], when
    ``fmt.has_act_scale``) into a new (or given) device blob."""
    N, K, G = fmt.N, fmt.K, fmt.G
    nbytes = packed_bytes(fmt)
    if nbytes == 0:
        _check("w4a16_pack", check_format(fmt))
    qp = _dev(q, torch.uint8, "q", (N, K))
    sp = _dev(scales, torch.float16, "scales", (N, G))
    zp = None if zeros is None else _dev(zeros, torch.uint8, "zeros", (N, G))
    ap = None if act_scale is None else _dev(act_scale, torch.float16, "act_scale", (K,))
    allocated = out is None
    if allocated:
        out = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    op = _dev(out, torch.uint8, "out")
    gi, gip = _host_gidx(g_idx, K)
    if fmt.has_act_scale:
        st = lib().w4a16_pack_awq(ctypes.byref(fmt), qp, sp, zp, gip, ap, op, out.numel(), _stream(stream))
        _check("w4a16_pack_awq", st)
    else:
        if ap is not None:
            raise ValueError("act_scale given but the format has no act scale")
        st = lib().w4a16_pack(ctypes.byref(fmt), qp, sp, zp, gip, op, out.numel(), _stream(stream))
        _check("w4a16_pack", st)
    if allocated:
        _keep_alive(stream, out)
    return out


def dequant(fmt: Format, packed: torch.Tensor, out: torch.Tensor | None = None, stream=None):
    pp = _dev(packed, torch.uint8, "packed")
    allocated = out is None
    if allocated:
        out = torch.empty((fmt.N, fmt.K), dtype=torch.float16, device=packed.device)
    op = _dev(out, torch.float16, "out", (fmt.N, fmt.K))
    _check("w4a16_dequant", lib().w4a16_dequant(ctypes.byref(fmt), pp, packed.numel(), op, _stream(stream)))
    if allocated:
        _keep_alive(stream, out)
    return out


GEMV_WEIGHTS_READY = 1
GEMV_REGISTER_RING = 2
GEMV_STAGE_ACTIVATIONS = 4
GEMV_ASYNC_COPY = 8
GEMV_INPUTS_READY = 16


def gemv(fmt: Format, packed: torch.Tensor, x: torch.Tensor, out: torch.Tensor | None = None,
         shape: int = 0, ksplit: int = 0, weights_ready: bool = False, register_ring: bool = False,
         stage_activations: bool = False, async_copy: bool = False, inputs_ready: bool = False,
         stream=None) -> torch.Tensor:
    """y = x . W_hat^T for x fp16 [M, K], 1 <= M <= 16.

    ``weights_ready``: the packed weights were complete before the previous
    kernel on the stream started, so the GEMV may stream them early.
    ``shape``: 16-row tiles per thread block. ``register_ring`` /
    ``async_copy``: force one of the two kernels (default: by layer size).
    ``stage_activations``: copy the activations to shared memory first.
    ``inputs_ready``: nothing in flight on the stream writes the weights or
    x or touches y, so the GEMV need not wait for the previous kernel.
    """
    M = x.shape[0]
    pp = _dev(packed, torch.uint8, "packed")
    xp = _dev(x, torch.float16, "x", (M, fmt.K))
    allocated = out is None
    if allocated:
        out = torch.empty((M, fmt.N), dtype=torch.float16, device=x.device)
    yp = _dev(out, torch.float16, "out", (M, fmt.N))
    flags = ((GEMV_WEIGHTS_READY if weights_ready else 0) | (GEMV_REGISTER_RING if register_ring else 0)
             | (GEMV_STAGE_ACTIVATIONS if stage_activations else 0) | (GEMV_ASYNC_COPY if async_copy else 0)
             | (GEMV_INPUTS_READY if inputs_ready else 0))
    if shape or ksplit or flags:
        st = lib().w4a16_gemv_ex(ctypes.byref(fmt), pp, packed.numel(), xp, yp, M, shape, ksplit, flags,
                                 _stream(stream))
    else:
        st = lib().w4a16_gemv(ctypes.byref(fmt), pp, packed.numel(), xp, yp, M, _stream(stream))
    _check("w4a16_gemv", st)
    if allocated:
        _keep_alive(stream, out)
    return out


def gemm_workspace_bytes(fmt: Format, M: int) -> int:
    return int(lib().w4a16_gemm_workspace_bytes(ctypes.byref(fmt), M))


def gemm(fmt: Format, packed: torch.Tensor, x: torch.Tensor, out: torch.Tensor | None = None,
         workspace: torch.Tensor | None = None, tile: int = 0, ksplit: int = 0, stream=None) -> torch.Tensor:
    """y = x . W_hat^T for x fp16 [M, K] on the tcgen05 tensor cores.

    ``tile`` / ``ksplit``: launch shape (0 = default), see ``w4a16_gemm_ex``.
    """
    M = x.shape[0]
    pp = _dev(packed, torch.uint8, "packed")
    xp = _dev(x, torch.float16, "x", (M, fmt.K))
    allocated = out is None
    if allocated:
        out = torch.empty((M, fmt.N), dtype=torch.float16, device=x.device)
    yp = _dev(out, torch.float16, "out", (M, fmt.N))
    need = gemm_workspace_bytes(fmt, M)
    own_ws = bool(need) and workspace is None
    if own_ws:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    wp = None if not need else _dev(workspace, torch.uint8, "workspace")
    wbytes = 0 if not need else workspace.numel()
    if tile or ksplit:
        st = lib().w4a16_gemm_ex(ctypes.byref(fmt), pp, packed.numel(), xp, yp, M, wp, wbytes, tile, ksplit,
                                 _stream(stream))
    else:
        st = lib().w4a16_gemm(ctypes.byref(fmt), pp, packed.numel(), xp, yp, M, wp, wbytes, _stream(stream))
    _check("w4a16_gemm", st)
    _keep_alive(stream, out if allocated else None, workspace if own_ws else None)
    return out


def pipeline_timeouts() -> int:
    """Bounded in-kernel waits that gave up on the current device since the last call (resets)."""
    c = ctypes.c_uint32(0)
    _check("w4a16_pipeline_timeouts", lib().w4a16_pipeline_timeouts(ctypes.byref(c)))
    return int(c.value)


def set_wait_limit_ns(ns: int) -> int:
    """Limit of the kernels' bounded waits for later launches (0: the 1 s default); returns the previous one."""
    return int(lib().w4a16_set_wait_limit_ns(int(ns)))


def debug_fail_next_launch(error: int) -> None:
    """Test hook: the next launching call returns W4A16_ERR_CUDA with this cudaError_t (0 clears)."""
    lib().w4a16_debug_fail_next_launch(int(error))


def debug_check_word():
    """First failed index check since the last call (0: none), read and reset;
    None when the loaded library is not the debug build."""
    w = ctypes.c_uint32(0)
    st = lib().w4a16_debug_check_word(ctypes.byref(w))
    if st == 2:  # W4A16_ERR_UNSUPPORTED: built without the checks
        return None
    _check("w4a16_debug_check_word", st)
    return int(w.value)


def linear(fmt: Format, packed: torch.Tensor, x: torch.Tensor, out=None, workspace=None, stream=None):
    """Dispatch by token count: the bandwidth-bound GEMV for M <= 16, else the GEMM."""
    if x.shape[0] <= 16:
        return gemv(fmt, packed, x, out=out, stream=stream)
    return gemm(fmt, packed, x, out=out, workspace=workspace, stream=stream)


class W4A16Linear:
    """A packed W4A16 linear layer resident in device memory."""

    def __init__(self, fmt: Format, packed: torch.Tensor):
        self.fmt = fmt
        self.packed = packed

    @classmethod
    def from_float(cls, w: torch.Tensor, group_size: int = 128, symmetric: bool = False, g_idx=None):
        """Quantize fp16 weights [N, K] (round to nearest) and pack them."""
        N, K = w.shape
        fmt = make_format(N, K, group_size, symmetric, g_idx is not None)
        q, s, z = quantize_rtn(fmt, w, g_idx)
        return cls(fmt, pack(fmt, q, s, z, g_idx))

    def __call__(self, x: torch.Tensor, out=None) -> torch.Tensor:
        return linear(self.fmt, self.packed, x, out=out)


class Chain:
    """A list of decode products run by one persistent launch (``w4a16_chain_*``).

    ``layers``: sequence of (fmt, packed, x, y, (wait_lo, wait_hi)) -- x fp16
    [M, K] and y fp16 [M, N] device tensors; the wait range names earlier
    layers whose outputs this layer reads (``None`` or an empty range: none).
    The tensors must stay alive as long as the chain is run.
    """

    def __init__(self, layers, M: int):
        n = len(layers)
        self.n = n
        fmts = (Format * n)()
        table = (ChainLayer * n)()
        keep = []
        for i, (fmt, packed, x, y, wait) in enumerate(layers):
            fmts[i] = fmt
            pp = _dev(packed, torch.uint8, "packed")
            xp = _dev(x, torch.float16, "x", (M, fmt.K))
            yp = _dev(y, torch.float16, "y", (M, fmt.N))
            lo, hi = (0, -1) if wait is None else wait
            table[i] = ChainLayer(pp, packed.numel(), xp, yp, lo, hi)
            keep.append((packed, x, y))
        self._keep = keep
        nbytes = int(lib().w4a16_chain_workspace_bytes(fmts, n, M))
        if nbytes == 0:
            raise ValueError("invalid or unsupported layer list for a chain")
        dev = layers[0][1].device
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.info = ChainInfo()
        st = lib().w4a16_chain_prepare(fmts, table, n, M, self.workspace.data_ptr(), nbytes,
                                       ctypes.byref(self.info))
        _check("w4a16_chain_prepare", st)

    def run(self, stream=None):
        st = lib().w4a16_chain_run(ctypes.byref(self.info), self.workspace.data_ptr(), _stream(stream))
        _check("w4a16_chain_run", st)
