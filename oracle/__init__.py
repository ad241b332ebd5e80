"""CPU oracle for the FP8 block-scaled linear (numpy front end over oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the product path never
does.  It shares no code with the CUDA library.  See ``oracle.c`` for the
passages each function follows and the readings taken where the pages are
silent.

Arrays: bf16 tensors travel as ``np.uint16`` bit patterns, e4m3 tensors as
``np.uint8`` codes, scales as ``np.float32``.

Parity status of each function (what pins it, see ``tests/test_oracle_*``):
  e4m3_decode / e4m3_encode   pinned (library codec, exhaustive decision points)
  bf16 conversions            pinned (library conversion)
  act_quant / weight_quant    pinned (zero / constant blocks, max code,
                              round-trip bounds, hand-derived worked example)
  weight_dequant              pinned (unit-scale closed form, library product)
  gemm / grouped_gemm         pinned (exact rational brute force, closed forms)
  silu_mul                    pinned (library silu, special values)
  moe_route / moe_combine     pinned (brute force, bincount, one-hot cases)
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32

BLOCK = 128


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.oracle_e4m3_decode.restype = ctypes.c_double
        L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        L.oracle_e4m3_encode_array.restype = None
        L.oracle_e4m3_encode_array.argtypes = [_f32p, _i64, _u8p]
        L.oracle_f32_to_bf16_array.restype = None
        L.oracle_f32_to_bf16_array.argtypes = [_f32p, _i64, _u16p]
        L.oracle_bf16_to_f32.restype = ctypes.c_float
        L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.oracle_f32_to_bf16.restype = ctypes.c_uint16
        L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        L.oracle_f64_to_bf16.restype = ctypes.c_uint16
        L.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
        L.oracle_pow2_ceil.restype = ctypes.c_float
        L.oracle_pow2_ceil.argtypes = [ctypes.c_float]
        L.oracle_act_quant.restype = None
        L.oracle_act_quant.argtypes = [_u16p, _i64, _i64, ctypes.c_int, _u8p, _f32p]
        L.oracle_weight_quant.restype = None
        L.oracle_weight_quant.argtypes = [_u16p, _i64, _i64, ctypes.c_int, _u8p, _f32p]
        L.oracle_weight_dequant.restype = None
        L.oracle_weight_dequant.argtypes = [_u8p, _f32p, _i64, _i64, _u16p]
        L.oracle_gemm.restype = None
        L.oracle_gemm.argtypes = [_u8p, _f32p, _u8p, _f32p, _i64, _i64, _i64,
                                  ctypes.c_void_p, _i64, _f64p, _f64p]
        L.oracle_grouped_gemm.restype = None
        L.oracle_grouped_gemm.argtypes = [_u8p, _f32p, _u8p, _f32p, _i32p, _i32, _i64, _i64,
                                          ctypes.c_void_p, _i64, _f64p, _f64p]
        L.oracle_silu_mul.restype = None
        L.oracle_silu_mul.argtypes = [_u16p, _u16p, _i64, _u16p]
        L.oracle_moe_route.restype = None
        L.oracle_moe_route.argtypes = [_i32p, _i64, _i32, _i32, _i32p, _i32p, _i32p]
        L.oracle_moe_combine.restype = None
        L.oracle_moe_combine.argtypes = [_u16p, _f32p, _i32p, _i64, _i32, _i64,
                                         ctypes.c_void_p, _i64, _f64p, _f64p]
        _lib = L
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- formats
def e4m3_decode(codes):
    """e4m3 codes (uint8) -> float64 values."""
    L = lib()
    table = np.array([L.oracle_e4m3_decode(c) for c in range(256)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(v):
    """float32 values -> e4m3 codes, RNE, saturating."""
    v = _c(v, np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().oracle_e4m3_encode_array(v.reshape(-1), v.size, out.reshape(-1))
    return out


def bf16_to_f32(h):
    h = np.asarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(f):
    """float32 -> bf16 bits, RNE."""
    f = _c(f, np.float32)
    out = np.empty(f.shape, dtype=np.uint16)
    lib().oracle_f32_to_bf16_array(f.reshape(-1), f.size, out.reshape(-1))
    return out


# ---------------------------------------------------------------- quantisation
def act_quant(x_bf16, ue8m0=False):
    """[DF "FP8 quantization data flow"] x: uint16 [M, K] -> (y uint8 [M, K], s f32 [M, K/128])."""
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    assert K % BLOCK == 0
    y = np.empty((M, K), dtype=np.uint8)
    s = np.empty((M, K // BLOCK), dtype=np.float32)
    lib().oracle_act_quant(x, M, K, int(bool(ue8m0)), y, s)
    return y, s


def weight_quant(w_bf16, ue8m0=False):
    """w: uint16 [N, K] -> (q uint8 [N, K], s f32 [ceil(N/128), ceil(K/128)])."""
    w = _c(w_bf16, np.uint16)
    N, K = w.shape
    q = np.empty((N, K), dtype=np.uint8)
    s = np.empty(((N + BLOCK - 1) // BLOCK, (K + BLOCK - 1) // BLOCK), dtype=np.float32)
    lib().oracle_weight_quant(w, N, K, int(bool(ue8m0)), q, s)
    return q, s


def weight_dequant(w_e4m3, s):
    """[BT "fp8->bf16 trace"] w: uint8 [M, N], s: f32 grid -> bf16 bits [M, N]."""
    w = _c(w_e4m3, np.uint8)
    s = _c(s, np.float32)
    M, N = w.shape
    assert s.shape == ((M + BLOCK - 1) // BLOCK, (N + BLOCK - 1) // BLOCK)
    y = np.empty((M, N), dtype=np.uint16)
    lib().oracle_weight_dequant(w, s, M, N, y)
    return y


# ---------------------------------------------------------------- GEMM
def _rows_arg(rows):
    if rows is None:
        return None, None
    r = np.ascontiguousarray(rows, dtype=np.int64)
    return r, r.ctypes.data_as(ctypes.c_void_p)


def gemm(a, a_s, b, b_s, rows=None):
    """Block-scaled product C = A B^T (exact, double).

    Returns (ref, mag) float64 [len(rows) or M, N]: ref the exact value, mag
    the same sum over absolute values."""
    a = _c(a, np.uint8); b = _c(b, np.uint8)
    a_s = _c(a_s, np.float32); b_s = _c(b_s, np.float32)
    M, K = a.shape
    N = b.shape[0]
    assert b.shape[1] == K and K % BLOCK == 0
    assert a_s.shape == (M, K // BLOCK)
    assert b_s.shape == ((N + BLOCK - 1) // BLOCK, K // BLOCK)
    r, rp = _rows_arg(rows)
    nrows = M if r is None else r.size
    if r is not None:
        assert np.all((r >= 0) & (r < M))
    ref = np.empty((nrows, N), dtype=np.float64)
    mag = np.empty((nrows, N), dtype=np.float64)
    lib().oracle_gemm(a, a_s, b, b_s, M, N, K, rp, nrows, ref, mag)
    return ref, mag


def grouped_gemm(a, a_s, b, b_s, offsets, rows=None):
    """Per-expert block-scaled product over packed rows (see oracle.c)."""
    a = _c(a, np.uint8); b = _c(b, np.uint8)
    a_s = _c(a_s, np.float32); b_s = _c(b_s, np.float32)
    offsets = _c(offsets, np.int32)
    G, N, K = b.shape
    assert offsets.shape == (G + 1,)
    r, rp = _rows_arg(rows)
    nrows = int(offsets[-1]) if r is None else r.size
    ref = np.empty((nrows, N), dtype=np.float64)
    mag = np.empty((nrows, N), dtype=np.float64)
    lib().oracle_grouped_gemm(a, a_s, b, b_s, offsets, G, N, K, rp, nrows, ref, mag)
    return ref, mag


def gemm_outputs(ref):
    """The kernel's two output forms for an exact result: fp32 (RN) and bf16
    (RNE of that fp32)."""
    f32 = np.asarray(ref, dtype=np.float64).astype(np.float32)
    return f32, f32_to_bf16(f32)


# ---------------------------------------------------------------- expert body / MoE
def silu_mul(h1, h3):
    h1 = _c(h1, np.uint16); h3 = _c(h3, np.uint16)
    assert h1.shape == h3.shape
    g = np.empty(h1.shape, dtype=np.uint16)
    lib().oracle_silu_mul(h1.reshape(-1), h3.reshape(-1), h1.size, g.reshape(-1))
    return g


def moe_route(ids, n_experts):
    """ids int32 [T, topk] -> (offsets [E+1], pair_row [T, topk], row_token [R])."""
    ids = _c(ids, np.int32)
    T, topk = ids.shape
    offsets = np.empty(n_experts + 1, dtype=np.int32)
    pair_row = np.empty((T, topk), dtype=np.int32)
    row_token = np.empty(T * topk, dtype=np.int32)
    lib().oracle_moe_route(ids.reshape(-1), T, topk, n_experts, offsets,
                           pair_row.reshape(-1), row_token)
    return offsets, pair_row, row_token


def moe_combine(out_bf16, weights, pair_row, tokens=None):
    """y[t] = sum_j w[t,j] * out[pair_row[t,j]] (double) -> (y, ymag)."""
    out = _c(out_bf16, np.uint16)
    w = _c(weights, np.float32)
    pr = _c(pair_row, np.int32)
    T, topk = w.shape
    D = out.shape[1]
    r, rp = _rows_arg(tokens)
    ntok = T if r is None else r.size
    y = np.empty((ntok, D), dtype=np.float64)
    ymag = np.empty((ntok, D), dtype=np.float64)
    lib().oracle_moe_combine(out, w, pr.reshape(-1), T, topk, D, rp, ntok, y, ymag)
    return y, ymag
