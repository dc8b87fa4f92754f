"""ctypes binding of libdr.so (include/dr.h).  Argument marshalling only: every
step of the forward and backward runs in the library's CUDA kernels; PyTorch
only allocates device memory and supplies the stream.

There is no fallback: if libdr.so is missing or a call fails, this module
raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdr.so")

DR_OK, DR_ERR_INVALID_ARG, DR_ERR_UNSUPPORTED, DR_ERR_WORKSPACE, DR_ERR_ALIGNMENT, \
    DR_ERR_CUDA, DR_ERR_TIMEOUT, DR_ERR_SCRATCH_LIMIT = range(8)
DR_DELTANET, DR_GDN, DR_KDA, DR_GDN2 = 0, 1, 2, 3
DR_BF16, DR_F32 = 0, 1
DR_FLAG_REUSE_FWD = 1
DR_FLAG_PREPARE_INPUTS = 2
VARIANTS = {"deltanet": DR_DELTANET, "gdn": DR_GDN, "kda": DR_KDA, "gdn2": DR_GDN2}


class DrDesc(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
        ("d_k", ctypes.c_int), ("d_v", ctypes.c_int), ("chunk", ctypes.c_int),
        ("variant", ctypes.c_int), ("io_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int),
        ("grad_dtype", ctypes.c_int), ("scale", ctypes.c_float), ("flags", ctypes.c_int),
        ("num_seqs", ctypes.c_int), ("cu_seqlens", ctypes.c_void_p),
        ("chunk_table", ctypes.c_void_p), ("chunk_offsets", ctypes.c_void_p),
        ("num_chunks", ctypes.c_int),
    ]


class DrError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {error_string(code)}")


_lib = None


def load(path: str = LIB_PATH):
    """Open libdr.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libdr.so not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    D = ctypes.POINTER(DrDesc)
    lib.dr_workspace_bytes.argtypes = [D]
    lib.dr_workspace_bytes.restype = S
    lib.dr_plan_varlen.argtypes = [P, I, I, P, P, I, P]
    lib.dr_plan_varlen.restype = I
    lib.dr_fwd.argtypes = [D] + [P] * 8 + [P, S, P]
    lib.dr_fwd.restype = I
    lib.dr_bwd.argtypes = [D] + [P] * 14 + [P, S, P]
    lib.dr_bwd.restype = I
    lib.dr_fwd_u.argtypes = [D] + [P] * 9 + [P, S, P]
    lib.dr_fwd_u.restype = I
    lib.dr_bwd_u.argtypes = [D] + [P] * 15 + [P, S, P]
    lib.dr_bwd_u.restype = I
    lib.dr_check_status.argtypes = [P, P]
    lib.dr_check_status.restype = I
    lib.dr_error_string.argtypes = [I]
    lib.dr_error_string.restype = ctypes.c_char_p
    lib.dr_fwd_noalloc.argtypes = [D] + [P] * 8 + [P]
    lib.dr_fwd_noalloc.restype = I
    lib.dr_decode.argtypes = [D] + [P] * 7 + [P]
    lib.dr_decode.restype = I
    lib.dr_gdn2_decode.argtypes = [D] + [P] * 8 + [P]
    lib.dr_gdn2_decode.restype = I
    lib.dr_selftest_wait.argtypes = [P, I, ctypes.c_longlong, P]
    lib.dr_selftest_wait.restype = I
    lib.dr_gdn2_fwd.argtypes = [D] + [P] * 9 + [P, S, P]
    lib.dr_gdn2_fwd.restype = I
    lib.dr_gdn2_bwd.argtypes = [D] + [P] * 16 + [P, S, P]
    lib.dr_gdn2_bwd.restype = I
    lib.dr_trace_enable.argtypes = [I]
    lib.dr_trace_enable.restype = I
    lib.dr_trace_count.argtypes = []
    lib.dr_trace_count.restype = I
    lib.dr_trace_reset.argtypes = []
    lib.dr_trace_reset.restype = None
    lib.dr_trace_get.argtypes = [I, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float)]
    lib.dr_trace_get.restype = I
    _lib = lib
    return lib


def error_string(code: int) -> str:
    return load().dr_error_string(int(code)).decode()


def _check(code: int, where: str):
    if code != DR_OK:
        raise DrError(code, where)


# ------------------------------------------------------------------ raw C-ABI calls
def workspace_bytes(desc: DrDesc) -> int:
    return int(load().dr_workspace_bytes(ctypes.byref(desc)))


def plan_varlen(cu_seqlens_host, chunk: int):
    """(chunk_table [n,2] int32, chunk_offsets [N+1] int32, n) for host offsets."""
    import numpy as np
    cu = np.ascontiguousarray(np.asarray(cu_seqlens_host, dtype=np.int32))
    N = len(cu) - 1
    n = ctypes.c_int(0)
    lib = load()
    _check(lib.dr_plan_varlen(cu.ctypes.data, N, chunk, None, None, 0, ctypes.byref(n)),
           "dr_plan_varlen")
    table = np.zeros((max(n.value, 1), 2), dtype=np.int32)
    offs = np.zeros(N + 1, dtype=np.int32)
    _check(lib.dr_plan_varlen(cu.ctypes.data, N, chunk, table.ctypes.data, offs.ctypes.data,
                              n.value, ctypes.byref(n)), "dr_plan_varlen")
    return table[:n.value], offs, n.value


def dr_fwd(desc, q, k, v, beta, g, h0, o, hT, ws, ws_bytes, stream) -> int:
    return load().dr_fwd(ctypes.byref(desc), q, k, v, beta, g, h0, o, hT, ws, ws_bytes, stream)


def dr_fwd_u(desc, q, k, v, beta, g, h0, o, hT, u, ws, ws_bytes, stream) -> int:
    return load().dr_fwd_u(ctypes.byref(desc), q, k, v, beta, g, h0, o, hT, u, ws, ws_bytes,
                           stream)


def dr_bwd_u(desc, q, k, v, beta, g, h0, dO, dhT, dU, dq, dk, dv, dbeta, dg, dh0, ws, ws_bytes,
             stream) -> int:
    return load().dr_bwd_u(ctypes.byref(desc), q, k, v, beta, g, h0, dO, dhT, dU, dq, dk, dv,
                           dbeta, dg, dh0, ws, ws_bytes, stream)


def dr_bwd(desc, q, k, v, beta, g, h0, dO, dhT, dq, dk, dv, dbeta, dg, dh0, ws, ws_bytes,
           stream) -> int:
    return load().dr_bwd(ctypes.byref(desc), q, k, v, beta, g, h0, dO, dhT, dq, dk, dv, dbeta,
                         dg, dh0, ws, ws_bytes, stream)


def dr_decode(desc, q, k, v, beta, g, state, o, stream) -> int:
    return load().dr_decode(ctypes.byref(desc), q, k, v, beta, g, state, o, stream)


def dr_gdn2_fwd(desc, q, k, v, erase, write, g, h0, o, hT, ws, ws_bytes, stream) -> int:
    return load().dr_gdn2_fwd(ctypes.byref(desc), q, k, v, erase, write, g, h0, o, hT, ws,
                              ws_bytes, stream)


def dr_gdn2_bwd(desc, q, k, v, erase, write, g, h0, dO, dhT, dq, dk, dv, derase, dwrite, dg, dh0,
                ws, ws_bytes, stream) -> int:
    return load().dr_gdn2_bwd(ctypes.byref(desc), q, k, v, erase, write, g, h0, dO, dhT, dq, dk,
                              dv, derase, dwrite, dg, dh0, ws, ws_bytes, stream)


def selftest_wait(ws, arrive: bool, limit_ns: int, stream) -> int:
    return load().dr_selftest_wait(ws, 1 if arrive else 0, int(limit_ns), stream)


def check_status(ws, stream) -> int:
    return load().dr_check_status(ws, stream)


def trace_enable(max_launches: int) -> None:
    _check(load().dr_trace_enable(int(max_launches)), "dr_trace_enable")


def trace_read():
    """[(kernel name, milliseconds)] of the traced launches, in launch order."""
    lib = load()
    out = []
    for i in range(lib.dr_trace_count()):
        name = ctypes.c_char_p()
        ms = ctypes.c_float()
        _check(lib.dr_trace_get(i, ctypes.byref(name), ctypes.byref(ms)), "dr_trace_get")
        out.append((name.value.decode(), float(ms.value)))
    return out


# ------------------------------------------------------------------ torch-level helpers
def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _dt(t) -> int:
    import torch
    return DR_BF16 if t.dtype == torch.bfloat16 else DR_F32


class Problem:
    """Descriptor + device-side chunk plan + workspace for one problem shape.

    Build once per shape; `forward` / `backward` then enqueue the library calls
    on the current torch stream.  With ``prepare`` the calls take raw q, k, beta
    logits and gate arguments (DR_FLAG_PREPARE_INPUTS) and the gradients are with
    respect to those.
    """

    def __init__(self, variant, B, T, H, dk, dv, chunk=64, io="bf16", out="f32",
                 grad="f32", scale=1.0, cu_seqlens=None, device="cuda", prepare=False):
        import torch
        self.device = torch.device(device)
        d = DrDesc()
        d.B, d.T, d.H, d.d_k, d.d_v, d.chunk = B, T, H, dk, dv, chunk
        d.variant = VARIANTS[variant] if isinstance(variant, str) else int(variant)
        code = {"bf16": DR_BF16, "f32": DR_F32}
        d.io_dtype, d.out_dtype, d.grad_dtype = code[io], code[out], code[grad]
        d.scale = float(scale)
        self.base_flags = DR_FLAG_PREPARE_INPUTS if prepare else 0
        d.flags = self.base_flags
        self._keep = []
        if cu_seqlens is not None:
            cu_host = [int(x) for x in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist")
                                        else cu_seqlens)]
            table, offs, n = plan_varlen(cu_host, chunk)
            cu_d = torch.tensor(cu_host, dtype=torch.int32, device=self.device)
            tab_d = torch.tensor(table.reshape(-1) if n else [0, 0], dtype=torch.int32,
                                 device=self.device)
            off_d = torch.tensor(offs, dtype=torch.int32, device=self.device)
            self._keep += [cu_d, tab_d, off_d]
            d.num_seqs = len(cu_host) - 1
            d.cu_seqlens, d.chunk_table, d.chunk_offsets = cu_d.data_ptr(), tab_d.data_ptr(), off_d.data_ptr()
            d.num_chunks = n
        else:
            d.num_seqs = B
            d.cu_seqlens = d.chunk_table = d.chunk_offsets = None
            d.num_chunks = 0
        self.desc = d
        self.N = d.num_seqs
        nbytes = workspace_bytes(d)
        if nbytes == 0:
            raise DrError(DR_ERR_UNSUPPORTED, "dr_workspace_bytes")
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        self.io_dtype = torch.bfloat16 if io == "bf16" else torch.float32
        self.out_dtype = torch.bfloat16 if out == "bf16" else torch.float32
        self.grad_dtype = torch.bfloat16 if grad == "bf16" else torch.float32

    def _stream(self):
        import torch
        return torch.cuda.current_stream(self.device).cuda_stream

    def forward(self, q, k, v, beta, g=None, h0=None, o=None, hT=None, want_hT=True, u=None):
        """o, hT; with `u` (a [B,T,H,dv] tensor of the output dtype) also the write
        beta r of every token (dr_fwd_u)."""
        import torch
        d = self.desc
        if o is None:
            o = torch.empty(d.B, d.T, d.H, d.d_v, dtype=self.out_dtype, device=self.device)
        if hT is None and want_hT:
            hT = torch.empty(self.N, d.H, d.d_k, d.d_v, dtype=torch.float32, device=self.device)
        if u is None:
            _check(dr_fwd(d, _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0), _ptr(o),
                          _ptr(hT), self.ws.data_ptr(), self.ws.numel(), self._stream()), "dr_fwd")
        else:
            _check(dr_fwd_u(d, _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0), _ptr(o),
                            _ptr(hT), _ptr(u), self.ws.data_ptr(), self.ws.numel(),
                            self._stream()), "dr_fwd_u")
        return o, hT

    def backward(self, q, k, v, beta, g, h0, dO, dhT=None, reuse_fwd=False, out=None, dU=None):
        import torch
        d = self.desc
        if out is None:
            out = {
                "dq": torch.empty(d.B, d.T, d.H, d.d_k, dtype=self.grad_dtype, device=self.device),
                "dk": torch.empty(d.B, d.T, d.H, d.d_k, dtype=self.grad_dtype, device=self.device),
                "dv": torch.empty(d.B, d.T, d.H, d.d_v, dtype=self.grad_dtype, device=self.device),
                "dbeta": torch.empty(d.B, d.T, d.H, dtype=torch.float32, device=self.device),
                "dg": None if g is None else torch.empty_like(g, dtype=torch.float32),
                "dh0": torch.empty(self.N, d.H, d.d_k, d.d_v, dtype=torch.float32,
                                   device=self.device),
            }
        d.flags = self.base_flags | (DR_FLAG_REUSE_FWD if reuse_fwd else 0)
        try:
            if dU is None:
                _check(dr_bwd(d, _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0),
                              _ptr(dO), _ptr(dhT), _ptr(out["dq"]), _ptr(out["dk"]),
                              _ptr(out["dv"]), _ptr(out["dbeta"]), _ptr(out["dg"]),
                              _ptr(out["dh0"]), self.ws.data_ptr(), self.ws.numel(),
                              self._stream()), "dr_bwd")
            else:
                _check(dr_bwd_u(d, _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0),
                                _ptr(dO), _ptr(dhT), _ptr(dU), _ptr(out["dq"]), _ptr(out["dk"]),
                                _ptr(out["dv"]), _ptr(out["dbeta"]), _ptr(out["dg"]),
                                _ptr(out["dh0"]), self.ws.data_ptr(), self.ws.numel(),
                                self._stream()), "dr_bwd_u")
        finally:
            d.flags = self.base_flags
        return out

    def status(self) -> int:
        return check_status(self.ws.data_ptr(), self._stream())


class Decoder:
    """Descriptor for the recurrent (token-by-token) step: `step` enqueues dr_decode
    on the current torch stream and updates `state` ([B, H, dk, dv] fp32) in place."""

    def __init__(self, variant, B, T, H, dk, dv, io="bf16", out="f32", scale=1.0,
                 device="cuda", prepare=False):
        import torch
        self.device = torch.device(device)
        d = DrDesc()
        d.B, d.T, d.H, d.d_k, d.d_v, d.chunk = B, T, H, dk, dv, 1
        d.variant = VARIANTS[variant] if isinstance(variant, str) else int(variant)
        code = {"bf16": DR_BF16, "f32": DR_F32}
        d.io_dtype, d.out_dtype, d.grad_dtype = code[io], code[out], code[out]
        d.scale = float(scale)
        d.flags = DR_FLAG_PREPARE_INPUTS if prepare else 0
        d.num_seqs = B
        d.cu_seqlens = d.chunk_table = d.chunk_offsets = None
        d.num_chunks = 0
        self.desc = d
        self.out_dtype = torch.bfloat16 if out == "bf16" else torch.float32

    def step(self, q, k, v, beta, g, state, o=None):
        import torch
        d = self.desc
        if o is None:
            o = torch.empty(d.B, d.T, d.H, d.d_v, dtype=self.out_dtype, device=self.device)
        _check(dr_decode(d, _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(state), _ptr(o),
                         torch.cuda.current_stream(self.device).cuda_stream), "dr_decode")
        return o

    def step_gdn2(self, q, k, v, erase, write, g, state, o=None):
        """Gated DeltaNet-2 (a Decoder built with variant "gdn2"): dr_gdn2_decode."""
        import torch
        d = self.desc
        if o is None:
            o = torch.empty(d.B, d.T, d.H, d.d_v, dtype=self.out_dtype, device=self.device)
        _check(load().dr_gdn2_decode(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(erase),
                                     _ptr(write), _ptr(g), _ptr(state), _ptr(o),
                                     torch.cuda.current_stream(self.device).cuda_stream),
               "dr_gdn2_decode")
        return o


class Gdn2Problem(Problem):
    """Gated DeltaNet-2 (dr_gdn2_fwd / dr_gdn2_bwd): the erase gate [B,T,H,dk] and the
    write gate [B,T,H,dv] take the place of beta."""

    def __init__(self, B, T, H, dk, dv, chunk=64, io="bf16", out="f32", grad="f32",
                 scale=1.0, cu_seqlens=None, device="cuda"):
        super().__init__("gdn2", B, T, H, dk, dv, chunk=chunk, io=io, out=out, grad=grad,
                         scale=scale, cu_seqlens=cu_seqlens, device=device)

    def forward(self, q, k, v, erase, write, g, h0=None, o=None, hT=None, want_hT=True):
        import torch
        d = self.desc
        if o is None:
            o = torch.empty(d.B, d.T, d.H, d.d_v, dtype=self.out_dtype, device=self.device)
        if hT is None and want_hT:
            hT = torch.empty(self.N, d.H, d.d_k, d.d_v, dtype=torch.float32, device=self.device)
        _check(dr_gdn2_fwd(d, _ptr(q), _ptr(k), _ptr(v), _ptr(erase), _ptr(write), _ptr(g),
                           _ptr(h0), _ptr(o), _ptr(hT), self.ws.data_ptr(), self.ws.numel(),
                           self._stream()), "dr_gdn2_fwd")
        return o, hT

    def backward(self, q, k, v, erase, write, g, h0, dO, dhT=None, out=None, reuse_fwd=False):
        import torch
        d = self.desc
        if out is None:
            f32 = dict(dtype=torch.float32, device=self.device)
            out = {
                "dq": torch.empty(d.B, d.T, d.H, d.d_k, dtype=self.grad_dtype, device=self.device),
                "dk": torch.empty(d.B, d.T, d.H, d.d_k, dtype=self.grad_dtype, device=self.device),
                "dv": torch.empty(d.B, d.T, d.H, d.d_v, dtype=self.grad_dtype, device=self.device),
                "derase": torch.empty(d.B, d.T, d.H, d.d_k, **f32),
                "dwrite": torch.empty(d.B, d.T, d.H, d.d_v, **f32),
                "dg": torch.empty(d.B, d.T, d.H, **f32),
                "dh0": torch.empty(self.N, d.H, d.d_k, d.d_v, **f32),
            }
        d.flags = DR_FLAG_REUSE_FWD if reuse_fwd else 0
        try:
            _check(dr_gdn2_bwd(d, _ptr(q), _ptr(k), _ptr(v), _ptr(erase), _ptr(write), _ptr(g),
                               _ptr(h0), _ptr(dO), _ptr(dhT), _ptr(out["dq"]), _ptr(out["dk"]),
                               _ptr(out["dv"]), _ptr(out["derase"]), _ptr(out["dwrite"]),
                               _ptr(out["dg"]), _ptr(out["dh0"]), self.ws.data_ptr(),
                               self.ws.numel(), self._stream()), "dr_gdn2_bwd")
        finally:
            d.flags = 0
        return out
