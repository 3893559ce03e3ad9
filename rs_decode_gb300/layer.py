"""Convenience owner of one layer's librs state, allocated as torch tensors.

The library allocates nothing; this class sizes every state array with
``rs_state_bytes_for`` and keeps the tensors alive.  Each method is one call
of the binding (which is one C entry point).  bf16 arrays are carried as int16
tensors holding the raw bit patterns.
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as rb


def to_device(d: dict, device="cuda", non_blocking: bool = False) -> dict:
    """numpy inputs (uint16 = bf16 bits, float32, int32) -> device tensors."""
    out = {}
    for k, v in d.items():
        a = np.ascontiguousarray(v)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        out[k] = torch.from_numpy(a).to(device, non_blocking=non_blocking)
    return out


class Layer:
    def __init__(self, kind: str, B: int, H: int, G: int, P: int, N: int, L: int, T_max: int = 0,
                 capacity: int | None = None, precision: int = rb.PREC_FP32, device="cuda"):
        if kind not in ("mamba2", "gdn", "kda"):
            raise ValueError(f"librs has no kernels for layer kind {kind!r}")
        self.kind = kind
        k = {"mamba2": rb.MAMBA2, "gdn": rb.GDN, "kda": rb.KDA}[kind]
        self.desc = rb.make_desc(k, B, H, G, P, N, L, T_max, capacity, precision)
        sz = rb.rs_state_bytes_for(self.desc)
        self.B, self.H, self.G, self.P, self.N, self.L, self.T_max = B, H, G, P, N, L, T_max
        self.cap = self.desc.capacity
        dev = torch.device(device)
        z = lambda n, dt: torch.zeros(n, dtype=dt, device=dev) if n else None
        self.ckpt_hp = z(sz.ckpt_hp // 4, torch.float32)
        self.ckpt_lp = z(sz.ckpt_lp // 2, torch.int16)
        self.buf_v = z(sz.buf_v, torch.uint8)
        self.buf_k = z(sz.buf_k // 2, torch.int16)
        self.buf_a = z(sz.buf_a // 4, torch.float32)
        self.buf_s = z(sz.buf_s // 4, torch.float32)
        self.base = z(B, torch.int32)
        self.h = z(B, torch.int32)
        self.nd = z(B, torch.int32)
        self.arrive = z(sz.arrive // 4, torch.int32)
        self.status_word = z(1, torch.int32)
        p = lambda t: t.data_ptr() if t is not None else None
        self.state = rb.State(p(self.ckpt_hp), p(self.ckpt_lp), p(self.buf_v), p(self.buf_k), p(self.buf_a),
                              p(self.buf_s), p(self.base), p(self.h), p(self.nd), p(self.arrive),
                              p(self.status_word))
        self.shape = (B, H, N, P)

    # ------------------------------------------------------------------ calls
    def init(self, S0: torch.Tensor | None = None, stream=None):
        """S0: fp32 [B, H, N, P] device tensor (key-major slabs) or None for zeros."""
        rb.rs_init(self.desc, self.state, S0, stream)

    def decode(self, d: dict, params: dict, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        if y is None:
            y = torch.empty(self.B, self.H, self.P, dtype=torch.float32, device=self.base.device)
        if self.kind == "mamba2":
            rb.rs_decode_mamba2(self.desc, self.state, d["x"], d["dt"], params["A"], d["Bm"], d["Cm"],
                                params.get("D"), y, stream)
        else:
            fn = rb.rs_decode_gdn if self.kind == "gdn" else rb.rs_decode_kda
            fn(self.desc, self.state, d["q"], d["k"], d["v"], d["alpha"], d["beta"], y, stream)
        return y

    def inputs(self, d: dict, params: dict) -> rb.Inputs:
        if self.kind == "mamba2":
            return rb.make_inputs(x=d["x"], dt=d["dt"], A=params["A"], Bm=d["Bm"], Cm=d.get("Cm"),
                                  D=params.get("D"))
        return rb.make_inputs(q=d["q"], k=d["k"], v=d["v"], alpha=d["alpha"], beta=d["beta"])

    def verify(self, T: int, d: dict, params: dict, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        if y is None:
            y = torch.empty(self.B, T, self.H, self.P, dtype=torch.float32, device=self.base.device)
        rb.rs_verify(self.desc, self.state, T, self.inputs(d, params), y, stream)
        return y

    def commit(self, accepted: torch.Tensor, stream=None):
        rb.rs_commit(self.desc, self.state, accepted, stream)

    def rollback(self, stream=None):
        rb.rs_rollback(self.desc, self.state, stream)

    def append(self, n: int, d: dict, params: dict, stream=None):
        rb.rs_append(self.desc, self.state, n, self.inputs(d, params), stream)

    def flush(self, stream=None):
        rb.rs_flush(self.desc, self.state, stream)

    def materialize(self, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty(self.shape, dtype=torch.float32, device=self.base.device)
        rb.rs_materialize(self.desc, self.state, out, stream)
        return out

    def status(self, clear: bool = True, stream=None) -> int:
        return rb.rs_get_status(self.state, clear, stream)

    def pointers(self) -> dict:
        return {"base": self.base.cpu().numpy(), "h": self.h.cpu().numpy(), "nd": self.nd.cpu().numpy()}

    def checkpoint_hp(self) -> torch.Tensor | None:
        return None if self.ckpt_hp is None else self.ckpt_hp.view(self.shape)

    def checkpoint_lp_f32(self) -> torch.Tensor | None:
        if self.ckpt_lp is None:
            return None
        return (self.ckpt_lp.to(torch.int32) << 16).view(torch.float32).view(self.shape)
