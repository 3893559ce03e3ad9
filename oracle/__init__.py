"""fp64 CPU oracle for the ReplaySSM decode path.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The CUDA
library never calls it, and it shares no code with the CUDA library: the
arithmetic lives in ``oracle.c`` (plain C, double precision, OpenMP over
(sequence, head)), compiled here with gcc.

What it computes is the conventional eager recurrence, which the method
reproduces apart from rounding ("ReplaySSM: Cache SSM Inputs,
Not State", sections "How it works" and "Limits"):

* Mamba-2: alpha_t = exp(dt_t A_h), S_t = alpha_t S_{t-1} + dt_t x_t k_t^T,
  y_t = S_t q_t + D_h x_t.
* Gated DeltaNet: u_t = beta_t (v_t - alpha_t S_{t-1} k_t),
  S_t = alpha_t S_{t-1} + u_t k_t^T, y_t = S_t q_t.
* Per-channel decay (a reading of Kimi Delta Attention, which section
  "Limits" names as compatible without defining it): GDN with the scalar decay
  replaced by one decay per key channel, D_t = S_{t-1} diag(alpha_t),
  u_t = beta_t (v_t - D_t k_t), S_t = D_t + u_t k_t^T, y_t = S_t q_t.
* Speculative round: the eager recurrence over the T drafts from the committed
  state; the state after the accepted prefix becomes the committed state.

State layout here is the mathematical one, S[b][h][p][n] (value index p,
key index n).  ``pointers`` models the checkpoint/buffer pointer rules so the
tests know when a flushed checkpoint must equal the eager state.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` with gcc (-O2 -fopenmp)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def use_library(path: str | None) -> None:
    """Load the oracle's functions from another build of ``oracle.c`` (the
    tests use this to check that their pins reject deliberately broken
    copies).  ``None`` returns to the default build."""
    global _lib, _path
    _lib, _path = None, path


_path = None


def _load():
    global _lib
    if _lib is None:
        if _path is None:
            build()
        lib = ctypes.CDLL(_path or _LIB)
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.oracle_mamba2_step.argtypes = [I, I, I, I, I] + [P] * 8
        lib.oracle_gdn_step.argtypes = [I, I, I, I, I] + [P] * 8
        lib.oracle_mamba2_spec_round.argtypes = [I, I, I, I, I, I] + [P] * 9
        lib.oracle_gdn_spec_round.argtypes = [I, I, I, I, I, I] + [P] * 8
        lib.oracle_kda_step.argtypes = [I, I, I, I, I] + [P] * 8
        lib.oracle_kda_spec_round.argtypes = [I, I, I, I, I, I] + [P] * 8
        lib.oracle_num_threads.restype = I
        _lib = lib
    return _lib


def _ptr(a: np.ndarray, dtype) -> int:
    assert a.dtype == dtype and a.flags["C_CONTIGUOUS"], (a.dtype, dtype)
    return a.ctypes.data


def num_threads() -> int:
    return _load().oracle_num_threads()


# ----------------------------------------------------------------------------- Mamba-2
def mamba2_step(S: np.ndarray, x, dt, A, Bm, Cm, D) -> np.ndarray:
    """One eager Mamba-2 step.  S f64[B,H,P,N] is updated in place.

    x u16[B,H,P] (bf16 bits), dt f32[B,H], A f32[H], Bm/Cm u16[B,G,N], D f32[H].
    Returns y f64[B,H,P].
    """
    B, H, P, N = S.shape
    G = Bm.shape[1]
    y = np.empty((B, H, P), np.float64)
    _load().oracle_mamba2_step(B, H, G, P, N, _ptr(S, np.float64), _ptr(x, np.uint16),
                               _ptr(dt, np.float32), _ptr(A, np.float32), _ptr(Bm, np.uint16),
                               _ptr(Cm, np.uint16), _ptr(D, np.float32), y.ctypes.data)
    return y


def mamba2_spec_round(S: np.ndarray, x, dt, A, Bm, Cm, D, accepted) -> np.ndarray:
    """One speculative round over T drafts.  Inputs carry a draft axis:
    x u16[B,T,H,P], dt f32[B,T,H], Bm/Cm u16[B,T,G,N], accepted i32[B].
    S (committed state) becomes the state after the accepted prefix.
    Returns y f64[B,T,H,P]."""
    B, H, P, N = S.shape
    T, G = x.shape[1], Bm.shape[2]
    y = np.empty((B, T, H, P), np.float64)
    _load().oracle_mamba2_spec_round(B, H, G, P, N, T, _ptr(S, np.float64), _ptr(x, np.uint16),
                                     _ptr(dt, np.float32), _ptr(A, np.float32),
                                     _ptr(Bm, np.uint16), _ptr(Cm, np.uint16),
                                     _ptr(D, np.float32), _ptr(accepted, np.int32), y.ctypes.data)
    return y


# ----------------------------------------------------------------------------- GDN
def gdn_step(S: np.ndarray, q, k, v, alpha, beta, want_u: bool = False):
    """One eager GDN step.  S f64[B,Hv,P,N] is updated in place.

    q, k u16[B,Hk,N]; v u16[B,Hv,P]; alpha, beta f32[B,Hv].
    Returns y f64[B,Hv,P] (and the correction term u f64[B,Hv,P] if asked).
    """
    B, Hv, P, N = S.shape
    Hk = q.shape[1]
    y = np.empty((B, Hv, P), np.float64)
    u = np.empty((B, Hv, P), np.float64) if want_u else None
    _load().oracle_gdn_step(B, Hv, Hk, P, N, _ptr(S, np.float64), _ptr(q, np.uint16),
                            _ptr(k, np.uint16), _ptr(v, np.uint16), _ptr(alpha, np.float32),
                            _ptr(beta, np.float32), y.ctypes.data,
                            u.ctypes.data if want_u else None)
    return (y, u) if want_u else y


def gdn_spec_round(S: np.ndarray, q, k, v, alpha, beta, accepted) -> np.ndarray:
    """One GDN speculative round; q, k u16[B,T,Hk,N], v u16[B,T,Hv,P],
    alpha, beta f32[B,T,Hv], accepted i32[B].  Returns y f64[B,T,Hv,P]."""
    B, Hv, P, N = S.shape
    T, Hk = q.shape[1], q.shape[2]
    y = np.empty((B, T, Hv, P), np.float64)
    _load().oracle_gdn_spec_round(B, Hv, Hk, P, N, T, _ptr(S, np.float64), _ptr(q, np.uint16),
                                  _ptr(k, np.uint16), _ptr(v, np.uint16), _ptr(alpha, np.float32),
                                  _ptr(beta, np.float32), _ptr(accepted, np.int32), y.ctypes.data)
    return y


# ----------------------------------------------------------------------------- per-channel decay
def kda_step(S: np.ndarray, q, k, v, alpha, beta, want_u: bool = False):
    """One eager step with a per-key-channel decay.  S f64[B,Hv,P,N] is
    updated in place.  q, k u16[B,Hk,N]; v u16[B,Hv,P]; alpha f32[B,Hv,N];
    beta f32[B,Hv].  Returns y f64[B,Hv,P] (and u f64[B,Hv,P] if asked)."""
    B, Hv, P, N = S.shape
    Hk = q.shape[1]
    assert alpha.shape == (B, Hv, N), alpha.shape
    y = np.empty((B, Hv, P), np.float64)
    u = np.empty((B, Hv, P), np.float64) if want_u else None
    _load().oracle_kda_step(B, Hv, Hk, P, N, _ptr(S, np.float64), _ptr(q, np.uint16),
                            _ptr(k, np.uint16), _ptr(v, np.uint16), _ptr(alpha, np.float32),
                            _ptr(beta, np.float32), y.ctypes.data,
                            u.ctypes.data if want_u else None)
    return (y, u) if want_u else y


def kda_spec_round(S: np.ndarray, q, k, v, alpha, beta, accepted) -> np.ndarray:
    """One speculative round with per-channel decays; q, k u16[B,T,Hk,N],
    v u16[B,T,Hv,P], alpha f32[B,T,Hv,N], beta f32[B,T,Hv], accepted i32[B].
    Returns y f64[B,T,Hv,P]."""
    B, Hv, P, N = S.shape
    T, Hk = q.shape[1], q.shape[2]
    assert alpha.shape == (B, T, Hv, N), alpha.shape
    y = np.empty((B, T, Hv, P), np.float64)
    _load().oracle_kda_spec_round(B, Hv, Hk, P, N, T, _ptr(S, np.float64), _ptr(q, np.uint16),
                                  _ptr(k, np.uint16), _ptr(v, np.uint16), _ptr(alpha, np.float32),
                                  _ptr(beta, np.float32), _ptr(accepted, np.int32), y.ctypes.data)
    return y


# ----------------------------------------------------------------------------- stateful model
class Model:
    """The eager recurrence for a batch of sequences of one layer, in fp64.

    ``kind`` is "mamba2", "gdn" or "kda"; ``S0`` f32/f64[B,H,P,N]; ``params`` holds
    A and D (Mamba-2).  ``step`` and ``spec_round`` take the input dicts that
    ``rs_decode_gb300.synth`` produces.
    """

    def __init__(self, kind: str, S0: np.ndarray, params: dict | None = None):
        if kind not in ("mamba2", "gdn", "kda"):
            raise ValueError(f"unknown layer kind {kind!r}")
        self.kind = kind
        self.S = np.array(S0, dtype=np.float64, order="C", copy=True)
        self.params = params or {}

    def step(self, d: dict) -> np.ndarray:
        if self.kind == "mamba2":
            return mamba2_step(self.S, d["x"], d["dt"], self.params["A"], d["Bm"], d["Cm"],
                               self.params["D"])
        step = gdn_step if self.kind == "gdn" else kda_step
        return step(self.S, d["q"], d["k"], d["v"], d["alpha"], d["beta"])

    def spec_round(self, d: dict) -> np.ndarray:
        if self.kind == "mamba2":
            return mamba2_spec_round(self.S, d["x"], d["dt"], self.params["A"], d["Bm"],
                                     d["Cm"], self.params["D"], d["accepted"])
        spec = gdn_spec_round if self.kind == "gdn" else kda_spec_round
        return spec(self.S, d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["accepted"])
