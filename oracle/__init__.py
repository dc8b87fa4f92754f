"""fp64 CPU oracle of the delta-rule recurrent memory (DeltaNet, Gated DeltaNet,
Kimi Delta Attention).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library never
does, and this package imports nothing from it.

The arithmetic lives in ``dro.c`` (a plain token-by-token loop in fp64, with the
hand-derived reverse-time recurrence for the gradients); this module only builds
it with gcc and marshals numpy arrays through ctypes.  What it computes is
defined on the page "Linear Attention Architectures: Mechanisms, Trade-offs, and
Cross-Layer Routing", section "Metodologia y Marco de Trabajo", item 1 (the
unified recurrent-memory notation and its DeltaNet / Gated DeltaNet / Kimi Delta
Attention bullets); the header of ``dro.c`` states each step.

``forward_gdn2`` / ``backward_gdn2`` run ``dro2.c``, the Gated DeltaNet-2 oracle (the
variant the same section describes in words only: separate erase and write gates per
channel); its header states the reading taken.  Pinned by ``tests/test_oracle_gdn2.py``
to that reading and, where they must agree, to the Gated DeltaNet oracle; the reading
itself is not fixed by the pages (parity of this variant is pinned to a reading).

Parity status: every other function here is pinned by ``tests/test_oracle.py``
(explicit matrix unrolling, central finite differences, the beta = 0 closed
form, exact recall, variant nesting, orthonormal keys, split/varlen chaining,
a hand-worked scalar example).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dro.c")
_SRC2 = os.path.join(_HERE, "dro2.c")
_LIB = os.path.join(_HERE, "libdro.so")
_lock = threading.Lock()
_lib = None

VARIANTS = {"deltanet": 0, "gdn": 1, "kda": 2}


def build(force: bool = False) -> str:
    """Compile dro.c and dro2.c into libdro.so (gcc, OpenMP if available)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= max(os.path.getmtime(_SRC), os.path.getmtime(_SRC2))):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c99", _SRC, _SRC2, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            common = [I, I, I, I, I, I, ctypes.c_double, P, I, P, I]
            lib.dro_forward.argtypes = common + [P] * 9 + [I]
            lib.dro_forward.restype = I
            lib.dro_backward.argtypes = common + [P] * 15 + [I]
            lib.dro_backward.restype = I
            common2 = [I, I, I, I, I, ctypes.c_double, P, I, P, I]
            lib.dro2_forward.argtypes = common2 + [P] * 9 + [I]
            lib.dro2_forward.restype = I
            lib.dro2_backward.argtypes = common2 + [P] * 16 + [I]
            lib.dro2_backward.restype = I
            lib.dro_max_threads.argtypes = []
            lib.dro_max_threads.restype = I
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().dro_max_threads())


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _i32(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def _dims(q, v, cu_seqlens):
    B, T, H, dk = q.shape
    dv = v.shape[3]
    N = B if cu_seqlens is None else len(cu_seqlens) - 1
    return B, T, H, dk, dv, N


def forward(variant, q, k, v, beta, g=None, h0=None, scale=1.0, cu_seqlens=None,
            units=None, nthreads=0, want_u=False):
    """Run the recurrence forward.  Returns (o, hT) as fp64 numpy arrays, or
    (o, hT, u) with ``want_u``: the write u_t = beta_t r_t, [B,T,H,dv].

    Shapes: q, k [B,T,H,dk]; v [B,T,H,dv]; beta [B,T,H]; g [B,T,H] (GDN) or
    [B,T,H,dk] (KDA) holding log(alpha); h0 [N,H,dk,dv] or None (zero state).
    ``units`` restricts the work to the listed (sequence*H + head) pairs; the
    other entries of the outputs stay zero.
    """
    vid = VARIANTS[variant] if isinstance(variant, str) else int(variant)
    q, k, v, beta, g, h0 = map(_f64, (q, k, v, beta, g, h0))
    cu = _i32(cu_seqlens)
    un = _i32(units)
    B, T, H, dk, dv, N = _dims(q, v, cu)
    o = np.zeros((B, T, H, dv))
    hT = np.zeros((N, H, dk, dv))
    u = np.zeros((B, T, H, dv)) if want_u else None
    rc = _load().dro_forward(B, T, H, dk, dv, vid, float(scale), _ptr(cu), N,
                             _ptr(un), 0 if un is None else len(un),
                             _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0),
                             _ptr(o), _ptr(hT), _ptr(u), int(nthreads))
    if rc != 0:
        raise ValueError("oracle forward: bad shape or arguments")
    return (o, hT, u) if want_u else (o, hT)


def backward(variant, q, k, v, beta, g, h0, dO, dhT=None, scale=1.0,
             cu_seqlens=None, units=None, nthreads=0, dU=None):
    """Reverse-time gradients of L = sum(dO*o) + sum(dhT*hT) (+ sum(dU*u) when dU,
    the gradient of the emitted write u, is given).  Returns dict dq, dk, dv,
    dbeta, dg (None for DeltaNet), dh0 (fp64 numpy)."""
    vid = VARIANTS[variant] if isinstance(variant, str) else int(variant)
    q, k, v, beta, g, h0, dO, dhT, dU = map(_f64, (q, k, v, beta, g, h0, dO, dhT, dU))
    cu = _i32(cu_seqlens)
    un = _i32(units)
    B, T, H, dk, dv, N = _dims(q, v, cu)
    dq = np.zeros_like(q)
    dk_ = np.zeros_like(k)
    dv_ = np.zeros_like(v)
    dbeta = np.zeros_like(beta)
    dg = None if vid == 0 else np.zeros_like(g)
    dh0 = np.zeros((N, H, dk, dv))
    rc = _load().dro_backward(B, T, H, dk, dv, vid, float(scale), _ptr(cu), N,
                              _ptr(un), 0 if un is None else len(un),
                              _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0),
                              _ptr(dO), _ptr(dhT), _ptr(dU), _ptr(dq), _ptr(dk_), _ptr(dv_),
                              _ptr(dbeta), _ptr(dg), _ptr(dh0), int(nthreads))
    if rc != 0:
        raise ValueError("oracle backward: bad shape or arguments")
    return {"dq": dq, "dk": dk_, "dv": dv_, "dbeta": dbeta, "dg": dg, "dh0": dh0}


def forward_gdn2(q, k, v, erase, write, g, h0=None, scale=1.0, cu_seqlens=None, units=None,
                 nthreads=0):
    """Gated DeltaNet-2 forward (dro2.c: scalar decay, per-key-channel erase gate,
    per-value-channel write gate).  Returns (o, hT) fp64.

    Shapes: q, k, erase [B,T,H,dk]; v, write [B,T,H,dv]; g [B,T,H] (log alpha);
    h0 [N,H,dk,dv] or None.
    """
    q, k, v, erase, write, g, h0 = map(_f64, (q, k, v, erase, write, g, h0))
    cu = _i32(cu_seqlens)
    un = _i32(units)
    B, T, H, dk, dv, N = _dims(q, v, cu)
    o = np.zeros((B, T, H, dv))
    hT = np.zeros((N, H, dk, dv))
    rc = _load().dro2_forward(B, T, H, dk, dv, float(scale), _ptr(cu), N, _ptr(un),
                              0 if un is None else len(un), _ptr(q), _ptr(k), _ptr(v),
                              _ptr(erase), _ptr(write), _ptr(g), _ptr(h0), _ptr(o), _ptr(hT),
                              int(nthreads))
    if rc != 0:
        raise ValueError("oracle forward_gdn2: bad shape or arguments")
    return o, hT


def backward_gdn2(q, k, v, erase, write, g, h0, dO, dhT=None, scale=1.0, cu_seqlens=None,
                  units=None, nthreads=0):
    """Gradients of L = sum(dO*o) + sum(dhT*hT) for Gated DeltaNet-2.  Returns dict
    dq, dk, dv, derase, dwrite, dg, dh0 (fp64)."""
    q, k, v, erase, write, g, h0, dO, dhT = map(_f64, (q, k, v, erase, write, g, h0, dO, dhT))
    cu = _i32(cu_seqlens)
    un = _i32(units)
    B, T, H, dk, dv, N = _dims(q, v, cu)
    out = {"dq": np.zeros_like(q), "dk": np.zeros_like(k), "dv": np.zeros_like(v),
           "derase": np.zeros_like(erase), "dwrite": np.zeros_like(write),
           "dg": np.zeros_like(g), "dh0": np.zeros((N, H, dk, dv))}
    rc = _load().dro2_backward(B, T, H, dk, dv, float(scale), _ptr(cu), N, _ptr(un),
                               0 if un is None else len(un), _ptr(q), _ptr(k), _ptr(v),
                               _ptr(erase), _ptr(write), _ptr(g), _ptr(h0), _ptr(dO), _ptr(dhT),
                               _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]),
                               _ptr(out["derase"]), _ptr(out["dwrite"]), _ptr(out["dg"]),
                               _ptr(out["dh0"]), int(nthreads))
    if rc != 0:
        raise ValueError("oracle backward_gdn2: bad shape or arguments")
    return out
