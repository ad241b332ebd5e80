"""GB300 (sm_103a) FP8 block-scaled linear: thin Python binding of the C ABI.

Every function here marshals torch tensors into the C entry point of the
same name declared in ``include/fp8bs.h`` and launches on the current CUDA
stream; all arithmetic runs in the library's kernels.  There is no CPU
fallback: importing this package fails if the shared library was not built
(``python fp8_block_scaled_07_gb300/_build.py`` or
``__graft_entry__.build()``), and every call raises :class:`Fp8Error` when
the library returns a non-OK status.

Tensors: bf16 as ``torch.bfloat16``; e4m3 as ``torch.float8_e4m3fn`` (a
``torch.uint8`` view of the same bytes is accepted); scales ``torch.float32``.
Outputs are allocated with torch (the caller's allocator) unless given.
"""
import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfp8bs.so")

FP8_SCALE_FP32 = 0
FP8_SCALE_UE8M0 = 1
BLOCK = 128

_STATUS = {0: "FP8_OK", 1: "FP8_ERR_INVALID_ARG", 2: "FP8_ERR_UNSUPPORTED", 3: "FP8_ERR_CUDA",
           4: "FP8_ERR_TIMEOUT", 5: "FP8_ERR_WORKSPACE"}


class Fp8Error(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn}: {_STATUS.get(status, status)} ({msg})")
        self.status = status


def _declare(lib):
    vp, i64, i32, f32p, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t
    st = ctypes.c_int
    sigs = {
        "fp8_act_quant": (st, [vp, vp, f32p, i64, i64, ctypes.c_int, vp]),
        "fp8_weight_quant": (st, [vp, vp, f32p, i64, i64, ctypes.c_int, vp]),
        "fp8_weight_dequant": (st, [vp, f32p, vp, i64, i64, vp]),
        "fp8_gemm_workspace_size": (sz, [i64, i64, i64]),
        "fp8_gemm": (st, [vp, f32p, vp, f32p, vp, f32p, i64, i64, i64, vp, sz, vp]),
        "fp8_gemm_ue8m0": (st, [vp, f32p, vp, f32p, vp, f32p, i64, i64, i64, vp]),
        "fp8_grouped_gemm": (st, [vp, f32p, vp, f32p, vp, i32, i64, vp, f32p, i64, i64, vp]),
        "fp8_silu_mul_quant": (st, [vp, vp, i64, i64, i64, vp, f32p, vp, ctypes.c_int, vp]),
        "fp8_moe_route": (st, [vp, i64, i32, i32, vp, vp, vp, vp]),
        "fp8_moe_gather": (st, [vp, f32p, vp, i64, i64, vp, f32p, vp]),
        "fp8_moe_combine": (st, [vp, f32p, vp, i64, i32, i64, vp, f32p, vp]),
        "fp8_linear_workspace_size": (sz, [i64, i64, i64]),
        "fp8_linear": (st, [vp, vp, f32p, vp, f32p, i64, i64, i64, ctypes.c_int, vp, sz, vp]),
        "fp8_gemm_noalloc": (st, [vp, f32p, vp, f32p, vp, f32p, i64, i64, i64, vp]),
        "fp8_gemm_swiglu": (st, [vp, f32p, vp, f32p, vp, f32p, i64, i64, i64, ctypes.c_int, vp]),
        "fp8_moe_expert_up": (st, [vp, f32p, vp, f32p, vp, i32, i64, vp, f32p, i64, i64, ctypes.c_int, vp]),
        "fp8_moe_quant_scatter": (st, [vp, vp, i64, i32, i64, vp, f32p, ctypes.c_int, vp]),
        "fp8_debug_set_wait_limit": (st, [ctypes.c_longlong]),
        "fp8_debug_skip_one_arrive": (None, []),
        "fp8_device_status": (st, [vp]),
        "fp8_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "fp8_num_sms": (ctypes.c_int, []),
    }
    for name, (res, args) in sigs.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            "fp8_block_scaled_07_gb300: native library %s is missing; build it with "
            "`python fp8_block_scaled_07_gb300/_build.py` (there is no CPU fallback)" % LIB_PATH)
    return _declare(ctypes.CDLL(LIB_PATH))


lib = _load()


# ------------------------------------------------------------------ helpers
# (kept light: a decode-sized call spends more time here than in the C entry)
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _ptr(t):
    return t.data_ptr() if t is not None else None   # c_void_p arguments take ints


def _stream(stream=None, device=None):
    """Raw cudaStream_t of `stream`, else of the current stream of `device`
    (an index; the current device if None)."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device() if device is None else device)
    return torch.cuda.current_stream().cuda_stream


def _check(name, status):
    if status != 0:
        raise Fp8Error(name, status, lib.fp8_status_string(status).decode())


def _cuda(t, name, dtypes, ndim=None):
    if (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype in dtypes and t.is_contiguous()
            and (ndim is None or t.dim() == ndim)):
        return t
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


_E4M3 = (torch.float8_e4m3fn, torch.uint8)
_BF16 = (torch.bfloat16,)
_F32 = (torch.float32,)
_I32 = (torch.int32,)


def _empty_e4m3(shape, device):
    return torch.empty(shape, dtype=torch.float8_e4m3fn, device=device)


# ------------------------------------------------------------------ ops
def fp8_act_quant(x, scale_fmt=FP8_SCALE_FP32, y=None, s=None, stream=None):
    """x [M, K] bf16 -> (y [M, K] e4m3, s [M, K/128] fp32)."""
    _cuda(x, "x", _BF16, 2)
    M, K = x.shape
    y = _empty_e4m3((M, K), x.device) if y is None else _cuda(y, "y", _E4M3)
    s = torch.empty((M, K // BLOCK), dtype=torch.float32, device=x.device) if s is None else _cuda(s, "s", _F32)
    _check("fp8_act_quant", lib.fp8_act_quant(_ptr(x), _ptr(y), _ptr(s), M, K, int(scale_fmt), _stream(stream)))
    return y, s


def fp8_weight_quant(w, scale_fmt=FP8_SCALE_FP32, q=None, s=None, stream=None):
    """w [N, K] bf16 -> (q [N, K] e4m3, s [ceil(N/128), ceil(K/128)] fp32)."""
    _cuda(w, "w", _BF16, 2)
    N, K = w.shape
    q = _empty_e4m3((N, K), w.device) if q is None else _cuda(q, "q", _E4M3)
    if s is None:
        s = torch.empty(((N + BLOCK - 1) // BLOCK, (K + BLOCK - 1) // BLOCK), dtype=torch.float32, device=w.device)
    _check("fp8_weight_quant", lib.fp8_weight_quant(_ptr(w), _ptr(q), _ptr(s), N, K, int(scale_fmt), _stream(stream)))
    return q, s


def fp8_weight_dequant(w, s, y=None, stream=None):
    """w [M, N] e4m3, s [ceil(M/128), ceil(N/128)] -> y [M, N] bf16."""
    _cuda(w, "w", _E4M3, 2)
    _cuda(s, "s", _F32, 2)
    M, N = w.shape
    if tuple(s.shape) != ((M + BLOCK - 1) // BLOCK, (N + BLOCK - 1) // BLOCK):
        raise ValueError("scale grid shape mismatch")
    y = torch.empty((M, N), dtype=torch.bfloat16, device=w.device) if y is None else _cuda(y, "y", _BF16)
    _check("fp8_weight_dequant", lib.fp8_weight_dequant(_ptr(w), _ptr(s), _ptr(y), M, N, _stream(stream)))
    return y


class _Workspace:
    """Zero-filled per-(device, stream) workspace, grown on demand.  The
    library leaves it zero-filled after every successful call."""

    def __init__(self):
        self._bufs = {}
        self._lock = threading.Lock()

    def get(self, nbytes, device, stream):
        """device: CUDA device index; stream: raw cudaStream_t of the call."""
        if nbytes == 0:
            return None
        key = (device, stream)
        buf = self._bufs.get(key)
        if buf is not None and buf.numel() >= nbytes:
            return buf
        with self._lock:
            buf = self._bufs.get(key)
            if buf is None or buf.numel() < nbytes:
                buf = torch.zeros(max(nbytes, 1 << 16), dtype=torch.uint8, device=torch.device("cuda", device))
                self._bufs[key] = buf
            return buf

    def reset(self):
        with self._lock:
            for b in self._bufs.values():
                b.zero_()


workspaces = _Workspace()


_ws_sizes = {}


def _ws_size(fn, M, N, K, device):
    """Workspace bytes of a call on `device` (an index), cached per shape: the
    plan depends only on the shape and the device's SM count."""
    key = (fn, M, N, K, device)
    v = _ws_sizes.get(key)
    if v is None:
        with torch.cuda.device(device):
            v = _ws_sizes[key] = int(getattr(lib, fn)(M, N, K))
    return v


def fp8_gemm_workspace_size(M, N, K):
    return int(lib.fp8_gemm_workspace_size(M, N, K))


def fp8_gemm(a, a_s, b, b_s, out_bf16=True, out_fp32=False, c_bf16=None, c_fp32=None,
             workspace=None, stream=None):
    """C = fp8 block-scaled a @ b^T.  Returns (c_bf16 or None, c_fp32 or None)."""
    _cuda(a, "a", _E4M3, 2)
    _cuda(b, "b", _E4M3, 2)
    _cuda(a_s, "a_s", _F32, 2)
    _cuda(b_s, "b_s", _F32, 2)
    M, K = a.shape
    N = b.shape[0]
    if b.shape[1] != K:
        raise ValueError("K mismatch")
    if tuple(a_s.shape) != (M, K // BLOCK) or tuple(b_s.shape) != ((N + BLOCK - 1) // BLOCK, K // BLOCK):
        raise ValueError("scale shape mismatch")
    if c_bf16 is None and out_bf16:
        c_bf16 = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    if c_fp32 is None and out_fp32:
        c_fp32 = torch.empty((M, N), dtype=torch.float32, device=a.device)
    st = _stream(stream)
    if workspace is None:
        dev = a.get_device()
        workspace = workspaces.get(_ws_size("fp8_gemm_workspace_size", M, N, K, dev), dev, st)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("fp8_gemm", lib.fp8_gemm(_ptr(a), _ptr(a_s), _ptr(b), _ptr(b_s), _ptr(c_bf16), _ptr(c_fp32),
                                    M, N, K, _ptr(workspace), ws_bytes, st))
    return c_bf16, c_fp32


def fp8_gemm_ue8m0(a, a_s, b, b_s, out_bf16=True, out_fp32=False, c_bf16=None, c_fp32=None, stream=None):
    """fp8_gemm for power-of-two (ue8m0) scales on the tensor core's block-scaled
    MMA.  Returns (c_bf16 or None, c_fp32 or None)."""
    _cuda(a, "a", _E4M3, 2)
    _cuda(b, "b", _E4M3, 2)
    _cuda(a_s, "a_s", _F32, 2)
    _cuda(b_s, "b_s", _F32, 2)
    M, K = a.shape
    N = b.shape[0]
    if b.shape[1] != K:
        raise ValueError("K mismatch")
    if tuple(a_s.shape) != (M, K // BLOCK) or tuple(b_s.shape) != ((N + BLOCK - 1) // BLOCK, K // BLOCK):
        raise ValueError("scale shape mismatch")
    if c_bf16 is None and out_bf16:
        c_bf16 = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    if c_fp32 is None and out_fp32:
        c_fp32 = torch.empty((M, N), dtype=torch.float32, device=a.device)
    _check("fp8_gemm_ue8m0", lib.fp8_gemm_ue8m0(_ptr(a), _ptr(a_s), _ptr(b), _ptr(b_s), _ptr(c_bf16),
                                                _ptr(c_fp32), M, N, K, _stream(stream)))
    return c_bf16, c_fp32


def fp8_grouped_gemm(a, a_s, b, b_s, offsets, out_bf16=True, out_fp32=False, c_bf16=None,
                     c_fp32=None, stream=None):
    """Per-expert fp8 GEMM over packed rows; offsets int32 [G+1] on the device."""
    _cuda(a, "a", _E4M3, 2)
    _cuda(b, "b", _E4M3, 3)
    _cuda(a_s, "a_s", _F32, 2)
    _cuda(b_s, "b_s", _F32, 3)
    _cuda(offsets, "offsets", _I32, 1)
    R, K = a.shape
    G, N, Kb = b.shape
    if Kb != K or offsets.numel() != G + 1:
        raise ValueError("shape mismatch")
    if c_bf16 is None and out_bf16:
        c_bf16 = torch.empty((R, N), dtype=torch.bfloat16, device=a.device)
    if c_fp32 is None and out_fp32:
        c_fp32 = torch.empty((R, N), dtype=torch.float32, device=a.device)
    _check("fp8_grouped_gemm", lib.fp8_grouped_gemm(_ptr(a), _ptr(a_s), _ptr(b), _ptr(b_s), _ptr(offsets),
                                                    G, R, _ptr(c_bf16), _ptr(c_fp32), N, K, _stream(stream)))
    return c_bf16, c_fp32


def interleave_w13(w1, w3, block=BLOCK):
    """Lay w1 and w3 ([I, K] each, or [G, I, K]) out as the fused kernels
    expect: 128-row blocks alternating w1, w3 -> [2I, K] (or [G, 2I, K]).
    Also for their scale grids ([I/128, K/128] -> [2I/128, K/128]) with
    block=1.  Pure data layout (a copy), no arithmetic."""
    if w1.shape != w3.shape:
        raise ValueError("w1 and w3 differ in shape")
    *lead, I, K = w1.shape
    if I % block:
        raise ValueError("rows not a multiple of the block")
    nb = I // block
    dt = w1.dtype
    if dt == torch.float8_e4m3fn:   # (moved as bytes)
        w1, w3 = w1.view(torch.uint8), w3.view(torch.uint8)
    a = w1.reshape(*lead, nb, block, K)
    b = w3.reshape(*lead, nb, block, K)
    return torch.stack([a, b], dim=-3).reshape(*lead, 2 * I, K).contiguous().view(dt)


def fp8_gemm_swiglu(a, a_s, w13, w13_s, scale_fmt=FP8_SCALE_FP32, g_q=None, g_s=None, stream=None):
    """act_quant(bf16(silu(h1)) * h3) with h1|h3 = a @ w13^T (w13 interleaved,
    see interleave_w13), in one GEMM launch.  Returns (g_q [M, I] e4m3,
    g_s [M, I/128] fp32)."""
    _cuda(a, "a", _E4M3, 2)
    _cuda(w13, "w13", _E4M3, 2)
    _cuda(a_s, "a_s", _F32, 2)
    _cuda(w13_s, "w13_s", _F32, 2)
    M, K = a.shape
    I = w13.shape[0] // 2
    if w13.shape[1] != K or tuple(w13_s.shape) != (2 * I // BLOCK, K // BLOCK):
        raise ValueError("shape mismatch")
    g_q = _empty_e4m3((M, I), a.device) if g_q is None else _cuda(g_q, "g_q", _E4M3)
    g_s = torch.empty((M, I // BLOCK), dtype=torch.float32, device=a.device) if g_s is None else _cuda(g_s, "g_s", _F32)
    _check("fp8_gemm_swiglu", lib.fp8_gemm_swiglu(_ptr(a), _ptr(a_s), _ptr(w13), _ptr(w13_s), _ptr(g_q), _ptr(g_s),
                                                  M, I, K, int(scale_fmt), _stream(stream)))
    return g_q, g_s


def fp8_moe_expert_up(a, a_s, w13, w13_s, offsets, scale_fmt=FP8_SCALE_FP32, g_q=None, g_s=None, stream=None):
    """Grouped w1|w3 + silu*mul + act_quant in one launch over packed rows.
    a [R, K] e4m3 / a_s [R, K/128]; w13 [G, 2I, K] interleaved (see
    interleave_w13); offsets int32 [G+1].  Returns (g_q [R, I], g_s [R, I/128])."""
    _cuda(a, "a", _E4M3, 2)
    _cuda(a_s, "a_s", _F32, 2)
    _cuda(w13, "w13", _E4M3, 3)
    _cuda(w13_s, "w13_s", _F32, 3)
    _cuda(offsets, "offsets", _I32, 1)
    R, K = a.shape
    G, N2, Kw = w13.shape
    I = N2 // 2
    if Kw != K or offsets.numel() != G + 1:
        raise ValueError("shape mismatch")
    g_q = _empty_e4m3((R, I), a.device) if g_q is None else g_q
    g_s = torch.empty((R, I // BLOCK), dtype=torch.float32, device=a.device) if g_s is None else g_s
    _check("fp8_moe_expert_up", lib.fp8_moe_expert_up(_ptr(a), _ptr(a_s), _ptr(w13), _ptr(w13_s), _ptr(offsets), G, R,
                                                      _ptr(g_q), _ptr(g_s), I, K, int(scale_fmt), _stream(stream)))
    return g_q, g_s


def fp8_moe_quant_scatter(x, pair_row, scale_fmt=FP8_SCALE_FP32, aq=None, as_=None, stream=None):
    """act_quant of x [T, K] bf16 written to the packed rows pair_row [T, topk]
    -> (aq [T*topk, K] e4m3, as [T*topk, K/128] fp32)."""
    _cuda(x, "x", _BF16, 2)
    _cuda(pair_row, "pair_row", _I32, 2)
    T, K = x.shape
    topk = pair_row.shape[1]
    R = T * topk
    aq = _empty_e4m3((R, K), x.device) if aq is None else aq
    as_ = torch.empty((R, K // BLOCK), dtype=torch.float32, device=x.device) if as_ is None else as_
    _check("fp8_moe_quant_scatter", lib.fp8_moe_quant_scatter(_ptr(x), _ptr(pair_row), T, topk, K, _ptr(aq),
                                                              _ptr(as_), int(scale_fmt), _stream(stream)))
    return aq, as_


def fp8_silu_mul_quant(h1, h3, ld_h, R, I, scale_fmt=FP8_SCALE_FP32, want_g=False, y=None, s=None,
                       stream=None):
    """g = bf16(bf16(silu(h1)) * h3) then act_quant(g).  h1/h3 are views into
    bf16 storage with row stride ld_h.  Returns (y, s, g or None)."""
    for name, t in (("h1", h1), ("h3", h3)):
        if not t.is_cuda or t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be a bf16 CUDA tensor")
    dev = h1.device
    y = _empty_e4m3((R, I), dev) if y is None else y
    s = torch.empty((R, I // BLOCK), dtype=torch.float32, device=dev) if s is None else s
    g = torch.empty((R, I), dtype=torch.bfloat16, device=dev) if want_g else None
    _check("fp8_silu_mul_quant", lib.fp8_silu_mul_quant(_ptr(h1), _ptr(h3), ld_h, R, I, _ptr(y), _ptr(s),
                                                        _ptr(g), int(scale_fmt), _stream(stream)))
    return y, s, g


def fp8_moe_route(ids, n_experts, stream=None):
    """ids int32 [T, topk] -> (offsets [E+1], pair_row [T, topk], row_token [T*topk])."""
    _cuda(ids, "ids", _I32, 2)
    T, topk = ids.shape
    offsets = torch.empty(n_experts + 1, dtype=torch.int32, device=ids.device)
    pair_row = torch.empty((T, topk), dtype=torch.int32, device=ids.device)
    row_token = torch.empty(T * topk, dtype=torch.int32, device=ids.device)
    _check("fp8_moe_route", lib.fp8_moe_route(_ptr(ids), T, topk, n_experts, _ptr(offsets), _ptr(pair_row),
                                              _ptr(row_token), _stream(stream)))
    return offsets, pair_row, row_token


def fp8_moe_gather(xq, xs, row_token, aq=None, as_=None, stream=None):
    _cuda(xq, "xq", _E4M3, 2)
    _cuda(xs, "xs", _F32, 2)
    _cuda(row_token, "row_token", _I32, 1)
    R = row_token.numel()
    K = xq.shape[1]
    aq = _empty_e4m3((R, K), xq.device) if aq is None else aq
    as_ = torch.empty((R, K // BLOCK), dtype=torch.float32, device=xq.device) if as_ is None else as_
    _check("fp8_moe_gather", lib.fp8_moe_gather(_ptr(xq), _ptr(xs), _ptr(row_token), R, K, _ptr(aq), _ptr(as_),
                                                _stream(stream)))
    return aq, as_


def fp8_moe_combine(out, w, pair_row, out_bf16=True, out_fp32=False, stream=None):
    _cuda(out, "out", _BF16, 2)
    _cuda(w, "w", _F32, 2)
    _cuda(pair_row, "pair_row", _I32, 2)
    T, topk = w.shape
    D = out.shape[1]
    yb = torch.empty((T, D), dtype=torch.bfloat16, device=out.device) if out_bf16 else None
    yf = torch.empty((T, D), dtype=torch.float32, device=out.device) if out_fp32 else None
    _check("fp8_moe_combine", lib.fp8_moe_combine(_ptr(out), _ptr(w), _ptr(pair_row), T, topk, D, _ptr(yb),
                                                  _ptr(yf), _stream(stream)))
    return yb, yf


def fp8_device_status(stream=None):
    """Synchronise and return the library's device status (raises on error)."""
    _check("fp8_device_status", lib.fp8_device_status(_stream(stream)))


def fp8_num_sms():
    return int(lib.fp8_num_sms())


def fp8_linear(x, w, w_s, scale_fmt=FP8_SCALE_FP32, out_bf16=True, out_fp32=False, c_bf16=None,
               c_fp32=None, workspace=None, stream=None):
    """The FP8 branch of the model's linear(): act_quant(x) then fp8_gemm, in
    one call (fused into one kernel for small decode batches).  Returns
    (c_bf16 or None, c_fp32 or None)."""
    _cuda(x, "x", _BF16, 2)
    _cuda(w, "w", _E4M3, 2)
    _cuda(w_s, "w_s", _F32, 2)
    M, K = x.shape
    N = w.shape[0]
    if w.shape[1] != K or tuple(w_s.shape) != ((N + BLOCK - 1) // BLOCK, K // BLOCK):
        raise ValueError("shape mismatch")
    if c_bf16 is None and out_bf16:
        c_bf16 = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    if c_fp32 is None and out_fp32:
        c_fp32 = torch.empty((M, N), dtype=torch.float32, device=x.device)
    st = _stream(stream)
    if workspace is None:
        dev = x.get_device()
        workspace = workspaces.get(_ws_size("fp8_linear_workspace_size", M, N, K, dev), dev, st)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("fp8_linear", lib.fp8_linear(_ptr(x), _ptr(w), _ptr(w_s), _ptr(c_bf16), _ptr(c_fp32), M, N, K,
                                        int(scale_fmt), _ptr(workspace), ws_bytes, st))
    return c_bf16, c_fp32
