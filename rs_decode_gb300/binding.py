"""Thin ctypes binding of librs (include/rs.h).

Argument marshalling only: every function here turns torch tensors into raw
pointers, passes the current CUDA stream, calls the C entry point of the same
name, and raises ``RsError`` on a non-zero status.  All arithmetic runs in the
library's CUDA kernels; there is no fallback of any kind, and loading fails
loudly when librs.so has not been built.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "librs.so")

MAMBA2, GDN, KDA = 0, 1, 2
PREC_FP32, PREC_TWO, PREC_SHARED_BF16 = 0, 1, 2
U_BF16 = 0x10  # flag: GDN records keep u in bf16
DEV_CAPACITY, DEV_ACCEPT, DEV_DRAFTS_PENDING = 0x1, 0x2, 0x4
STATUS = {0: "RS_OK", 1: "RS_ERR_INVALID_ARG", 2: "RS_ERR_UNSUPPORTED", 3: "RS_ERR_CAPACITY",
          4: "RS_ERR_CUDA", 5: "RS_ERR_DEVICE", 6: "RS_ERR_STATIC_LIMIT"}
STATIC_MAX_SEQS = 4096

_c_i32 = ctypes.c_int32
_vp = ctypes.c_void_p


class LayerDesc(ctypes.Structure):
    _fields_ = [(n, _c_i32) for n in ("kind", "B", "H", "G", "P", "N", "L", "T_max", "capacity",
                                       "precision")]


class State(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("ckpt_hp", "ckpt_lp", "buf_v", "buf_k", "buf_a", "buf_s", "base",
                                    "h", "nd", "arrive", "status")]


class StateBytes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("ckpt_hp", "ckpt_lp", "buf_v", "buf_k", "buf_a",
                                                "buf_s", "base", "h", "nd", "arrive", "status")]


class Inputs(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("x", "dt", "A", "Bm", "Cm", "D", "q", "k", "v", "alpha", "beta")]


# name -> argtypes (restype is rs_status = int unless listed in _RESTYPE)
_SIGS = {
    "rs_status_string": [ctypes.c_int],
    "rs_version": [],
    "rs_last_cuda_error": [],
    "rs_state_bytes_for": [ctypes.POINTER(LayerDesc), ctypes.POINTER(StateBytes)],
    "rs_init": [ctypes.POINTER(LayerDesc), ctypes.POINTER(State), _vp, _vp],
    "rs_get_status": [ctypes.POINTER(State), ctypes.POINTER(ctypes.c_uint32), ctypes.c_int, _vp],
    "rs_decode_mamba2": [ctypes.POINTER(LayerDesc), ctypes.POINTER(State)] + [_vp] * 8,
    "rs_decode_gdn": [ctypes.POINTER(LayerDesc), ctypes.POINTER(State)] + [_vp] * 7,
    "rs_decode_kda": [ctypes.POINTER(LayerDesc), ctypes.POINTER(State)] + [_vp] * 7,
    "rs_verify": [ctypes.POINTER(LayerDesc), ctypes.POINTER(State), ctypes.c_int,
                  ctypes.POINTER(Inputs), _vp, _vp],
    "rs_commit": [ctypes.POINTER(LayerDesc), ctypes.POINTER(State), _vp, _vp],
    "rs_rollback": [ctypes.POINTER(LayerDesc), ctypes.POINTER(State), _vp],
    "rs_append": [ctypes.POINTER(LayerDesc), ctypes.POINTER(State), ctypes.c_int,
                  ctypes.POINTER(Inputs), _vp],
    "rs_flush": [ctypes.POINTER(LayerDesc), ctypes.POINTER(State), _vp],
    "rs_materialize": [ctypes.POINTER(LayerDesc), ctypes.POINTER(State), _vp, _vp],
    "rs_eager_step_mamba2": [ctypes.POINTER(LayerDesc)] + [_vp] * 9,
    "rs_eager_step_gdn": [ctypes.POINTER(LayerDesc)] + [_vp] * 8,
    "rs_eager_step_kda": [ctypes.POINTER(LayerDesc)] + [_vp] * 8,
    "rs_eager_verify_snapshots": [ctypes.POINTER(LayerDesc), _vp, _vp, ctypes.c_int,
                                  ctypes.POINTER(Inputs), _vp, _vp],
    "rs_eager_select": [ctypes.POINTER(LayerDesc), _vp, _vp, _vp, _vp],
    "rs_decode_mamba2_noalloc": [ctypes.POINTER(LayerDesc), ctypes.POINTER(State)] + [_vp] * 8,
}
_RESTYPE = {"rs_status_string": ctypes.c_char_p, "rs_version": ctypes.c_char_p,
            "rs_last_cuda_error": ctypes.c_char_p}

_lib = None


class RsError(RuntimeError):
    def __init__(self, fn: str, status: int, bits: int | None = None):
        self.status = status
        self.bits = bits
        extra = f" (device bits 0x{bits:x})" if bits is not None else ""
        super().__init__(f"{fn} returned {STATUS.get(status, status)}{extra}")


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load librs.so (no GPU needed).  Raises if the library was not built."""
    global _lib
    if _lib is None or path != LIB_PATH:
        if not os.path.exists(path):
            raise RuntimeError(f"librs.so not found at {path}: run rs_decode_gb300.build.build() "
                               "(or __graft_entry__.build()) first")
        lib = ctypes.CDLL(path)
        for name, args in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = _RESTYPE.get(name, ctypes.c_int)
        if path != LIB_PATH:
            return lib
        _lib = lib
    return _lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensors passed to librs must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _check(fn: str, status: int) -> None:
    if status != 0:
        err = RsError(fn, status)
        if status == 4:  # RS_ERR_CUDA: say which CUDA error
            err.args = (f"{err.args[0]}: {load().rs_last_cuda_error().decode()}",)
        raise err


def make_desc(kind: int, B: int, H: int, G: int, P: int, N: int, L: int, T_max: int = 0,
              capacity: int | None = None, precision: int = PREC_FP32) -> LayerDesc:
    return LayerDesc(kind, B, H, G, P, N, L, T_max, capacity if capacity else max(L, T_max) + T_max, precision)


# Precision names of the synthetic workloads: the checkpoint's, and "+u16"
# for GDN records that keep u in bf16.
PRECISIONS = {"fp32": PREC_FP32, "two": PREC_TWO, "shared_bf16": PREC_SHARED_BF16,
              "fp32+u16": PREC_FP32 | U_BF16, "two+u16": PREC_TWO | U_BF16}


def make_inputs(**tensors) -> Inputs:
    return Inputs(**{k: _ptr(v) for k, v in tensors.items() if v is not None})


# ----------------------------------------------------------------------------- entry points
def rs_version() -> str:
    return load().rs_version().decode()


def rs_status_string(status: int) -> str:
    return load().rs_status_string(status).decode()


def rs_state_bytes_for(desc: LayerDesc) -> StateBytes:
    out = StateBytes()
    _check("rs_state_bytes_for", load().rs_state_bytes_for(ctypes.byref(desc), ctypes.byref(out)))
    return out


def rs_init(desc, state, init=None, stream=None):
    _check("rs_init", load().rs_init(ctypes.byref(desc), ctypes.byref(state), _ptr(init), _stream(stream)))


def rs_get_status(state, clear: bool = True, stream=None) -> int:
    bits = ctypes.c_uint32(0)
    st = load().rs_get_status(ctypes.byref(state), ctypes.byref(bits), int(clear), _stream(stream))
    if st not in (0, 5):
        raise RsError("rs_get_status", st)
    return bits.value


def rs_decode_mamba2(desc, state, x, dt, A, Bm, Cm, D, y, stream=None):
    _check("rs_decode_mamba2", load().rs_decode_mamba2(
        ctypes.byref(desc), ctypes.byref(state), _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm),
        _ptr(D), _ptr(y), _stream(stream)))


def rs_decode_gdn(desc, state, q, k, v, alpha, beta, y, stream=None):
    _check("rs_decode_gdn", load().rs_decode_gdn(
        ctypes.byref(desc), ctypes.byref(state), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
        _ptr(y), _stream(stream)))


def rs_decode_kda(desc, state, q, k, v, alpha, beta, y, stream=None):
    _check("rs_decode_kda", load().rs_decode_kda(
        ctypes.byref(desc), ctypes.byref(state), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
        _ptr(y), _stream(stream)))


def rs_verify(desc, state, T: int, inputs: Inputs, y, stream=None):
    _check("rs_verify", load().rs_verify(ctypes.byref(desc), ctypes.byref(state), T,
                                         ctypes.byref(inputs), _ptr(y), _stream(stream)))


def rs_commit(desc, state, accepted, stream=None):
    _check("rs_commit", load().rs_commit(ctypes.byref(desc), ctypes.byref(state), _ptr(accepted),
                                         _stream(stream)))


def rs_rollback(desc, state, stream=None):
    _check("rs_rollback", load().rs_rollback(ctypes.byref(desc), ctypes.byref(state), _stream(stream)))


def rs_append(desc, state, n: int, inputs: Inputs, stream=None):
    _check("rs_append", load().rs_append(ctypes.byref(desc), ctypes.byref(state), n,
                                         ctypes.byref(inputs), _stream(stream)))


def rs_flush(desc, state, stream=None):
    _check("rs_flush", load().rs_flush(ctypes.byref(desc), ctypes.byref(state), _stream(stream)))


def rs_materialize(desc, state, out, stream=None):
    _check("rs_materialize", load().rs_materialize(ctypes.byref(desc), ctypes.byref(state), _ptr(out),
                                                   _stream(stream)))


def rs_eager_step_mamba2(desc, S, x, dt, A, Bm, Cm, D, y, stream=None):
    _check("rs_eager_step_mamba2", load().rs_eager_step_mamba2(
        ctypes.byref(desc), _ptr(S), _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm), _ptr(D), _ptr(y),
        _stream(stream)))


def rs_eager_step_gdn(desc, S, q, k, v, alpha, beta, y, stream=None):
    _check("rs_eager_step_gdn", load().rs_eager_step_gdn(
        ctypes.byref(desc), _ptr(S), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(y),
        _stream(stream)))


def rs_eager_step_kda(desc, S, q, k, v, alpha, beta, y, stream=None):
    _check("rs_eager_step_kda", load().rs_eager_step_kda(
        ctypes.byref(desc), _ptr(S), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(y),
        _stream(stream)))


def rs_eager_verify_snapshots(desc, pool, cur, T: int, inputs: Inputs, y, stream=None):
    _check("rs_eager_verify_snapshots", load().rs_eager_verify_snapshots(
        ctypes.byref(desc), _ptr(pool), _ptr(cur), T, ctypes.byref(inputs), _ptr(y), _stream(stream)))


def rs_eager_select(desc, cur, accepted, status=None, stream=None):
    _check("rs_eager_select", load().rs_eager_select(ctypes.byref(desc), _ptr(cur), _ptr(accepted),
                                                     _ptr(status), _stream(stream)))


def rs_decode_mamba2_noalloc(desc, state, x, dt, A, Bm, Cm, D, y, stream=None):
    """rs_decode_mamba2 with the arrival counters in the library's static
    device array (state.arrive is ignored); for callers that cannot allocate."""
    _check("rs_decode_mamba2_noalloc", load().rs_decode_mamba2_noalloc(
        ctypes.byref(desc), ctypes.byref(state), _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm),
        _ptr(D), _ptr(y), _stream(stream)))
