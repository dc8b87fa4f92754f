"""Host-side checks of the C ABI (no GPU needed, no kernel is launched):
the library loads, exports every entry point of include/dr.h, and rejects bad
arguments with the documented codes before touching the device."""
import ctypes
import os
import re

import numpy as np
import pytest

from delta_rule_recurrent_gated_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from delta_rule_recurrent_gated_gb300 import build
    build.build()
    return B.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "dr.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dr_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"dr_fwd", "dr_bwd", "dr_workspace_bytes", "dr_plan_varlen", "dr_check_status",
            "dr_error_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in dr.h but not exported"


def desc(**kw):
    d = B.DrDesc()
    d.B, d.T, d.H, d.d_k, d.d_v, d.chunk = 2, 128, 4, 128, 128, 64
    d.variant, d.io_dtype, d.out_dtype, d.grad_dtype = B.DR_GDN, B.DR_BF16, B.DR_F32, B.DR_F32
    d.scale, d.flags, d.num_seqs = 1.0, 0, 2
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def test_struct_layout_matches_header(lib, tmp_path):
    """The binding's dr_desc must agree field by field with the C compiler's."""
    import shutil
    import subprocess
    if not shutil.which("gcc"):
        pytest.skip("gcc not available")
    names = [f[0] for f in B.DrDesc._fields_]
    src = tmp_path / "layout.c"
    body = "".join(f'printf("%zu\\n", offsetof(dr_desc, {n}));' for n in names)
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "dr.h"\n'
                   'int main(void){' + body + 'printf("%zu\\n", sizeof(dr_desc));return 0;}\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    out = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    assert out[:-1] == [getattr(B.DrDesc, n).offset for n in names]
    assert out[-1] == ctypes.sizeof(B.DrDesc)


def test_workspace_bytes(lib):
    assert B.workspace_bytes(desc()) > 0
    assert B.workspace_bytes(desc(io_dtype=B.DR_F32, d_k=32, d_v=32, chunk=16)) > 0
    assert B.workspace_bytes(desc(H=0)) == 0
    assert B.workspace_bytes(desc(d_k=96, d_v=96)) == 0          # unsupported
    assert B.workspace_bytes(desc(chunk=32)) == 0                 # bf16 path needs chunk 64
    # the fp32 CUDA-core path takes d_k, d_v up to 128 (chunk at most 64)
    assert B.workspace_bytes(desc(io_dtype=B.DR_F32, d_k=128, d_v=128, chunk=64)) > 0
    assert B.workspace_bytes(desc(io_dtype=B.DR_F32, d_k=128, d_v=16, chunk=16)) > 0
    assert B.workspace_bytes(desc(io_dtype=B.DR_F32, d_k=96, d_v=96, chunk=64)) == 0
    assert B.workspace_bytes(desc(io_dtype=B.DR_F32, d_k=128, d_v=128, chunk=128)) == 0


def call_fwd(d, ptrs=None, ws=None, ws_bytes=1 << 40):
    p = dict(q=16, k=16, v=16, beta=16, g=16, h0=None, o=16, hT=None)
    if ptrs:
        p.update(ptrs)
    return B.dr_fwd(d, p["q"], p["k"], p["v"], p["beta"], p["g"], p["h0"], p["o"], p["hT"],
                    16 if ws is None else ws, ws_bytes, None)


def test_fwd_argument_errors(lib):
    assert call_fwd(desc(variant=7)) == B.DR_ERR_INVALID_ARG
    assert call_fwd(desc(B=-1)) == B.DR_ERR_INVALID_ARG
    assert call_fwd(desc(io_dtype=5)) == B.DR_ERR_INVALID_ARG
    assert call_fwd(desc(scale=float("nan"))) == B.DR_ERR_INVALID_ARG
    assert call_fwd(desc(flags=8)) == B.DR_ERR_INVALID_ARG
    assert call_fwd(desc(num_seqs=3)) == B.DR_ERR_INVALID_ARG      # dense: N must equal B
    assert call_fwd(desc(), ptrs={"q": None}) == B.DR_ERR_INVALID_ARG
    assert call_fwd(desc(), ptrs={"g": None}) == B.DR_ERR_INVALID_ARG       # GDN needs g
    assert call_fwd(desc(variant=B.DR_DELTANET)) == B.DR_ERR_INVALID_ARG    # DeltaNet: g NULL
    assert call_fwd(desc(d_k=96, d_v=96)) == B.DR_ERR_UNSUPPORTED
    assert call_fwd(desc(), ptrs={"k": 24}) == B.DR_ERR_ALIGNMENT
    assert call_fwd(desc(), ptrs={"hT": 8}) == B.DR_ERR_ALIGNMENT
    assert call_fwd(desc(), ws=0) == B.DR_ERR_WORKSPACE
    assert call_fwd(desc(), ws_bytes=100) == B.DR_ERR_WORKSPACE
    # packed layout needs B == 1 and the chunk tables
    assert call_fwd(desc(B=2, cu_seqlens=16, num_seqs=2, chunk_offsets=16)) == B.DR_ERR_INVALID_ARG
    assert call_fwd(desc(B=1, cu_seqlens=16, num_seqs=2, num_chunks=3,
                         chunk_offsets=16)) == B.DR_ERR_INVALID_ARG


def test_bwd_argument_errors(lib):
    def bwd(d, **kw):
        p = dict(q=16, k=16, v=16, beta=16, g=16, h0=None, dO=16, dhT=None, dq=16, dk=16,
                 dv=16, dbeta=16, dg=16, dh0=None)
        p.update(kw)
        return B.dr_bwd(d, *p.values(), 16, 1 << 40, None)
    assert bwd(desc(), dO=None) == B.DR_ERR_INVALID_ARG
    assert bwd(desc(), dg=None) == B.DR_ERR_INVALID_ARG
    assert bwd(desc(variant=B.DR_DELTANET), g=None) == B.DR_ERR_INVALID_ARG  # dg must be NULL
    assert bwd(desc(), dh0=4) == B.DR_ERR_ALIGNMENT
    assert bwd(desc(d_k=64, d_v=128)) == B.DR_ERR_UNSUPPORTED


def test_error_strings(lib):
    for c in range(7):
        assert B.error_string(c).startswith("DR_")
    assert "unknown" in B.error_string(99)


def python_plan(cu, chunk):
    table, offs = [], []
    for n in range(len(cu) - 1):
        offs.append(len(table))
        t = cu[n]
        while t < cu[n + 1]:
            table.append((n, t))
            t += chunk
    offs.append(len(table))
    return table, offs


@pytest.mark.parametrize("lens", [[5], [64], [65, 0, 130, 1], [0, 0], [256, 4000, 33, 64, 63]])
@pytest.mark.parametrize("chunk", [16, 64])
def test_plan_varlen_is_exact(lib, lens, chunk):
    cu = np.cumsum([0] + lens).astype(np.int32)
    table, offs, n = B.plan_varlen(cu, chunk)
    rt, ro = python_plan(cu.tolist(), chunk)
    assert n == len(rt)
    assert table.tolist() == [list(x) for x in rt]
    assert offs.tolist() == ro
    # every token covered exactly once, no chunk straddles a boundary
    cover = np.zeros(cu[-1], dtype=np.int32)
    for s, t0 in table:
        end = min(t0 + chunk, cu[s + 1])
        assert cu[s] <= t0 < cu[s + 1]
        cover[t0:end] += 1
    assert np.all(cover == 1)


def test_plan_varlen_errors(lib):
    n = ctypes.c_int(0)
    bad = np.array([1, 5], dtype=np.int32)
    assert lib.dr_plan_varlen(bad.ctypes.data, 1, 64, None, None, 0, ctypes.byref(n)) == B.DR_ERR_INVALID_ARG
    dec = np.array([0, 9, 4], dtype=np.int32)
    assert lib.dr_plan_varlen(dec.ctypes.data, 2, 64, None, None, 0, ctypes.byref(n)) == B.DR_ERR_INVALID_ARG
    ok = np.array([0, 200], dtype=np.int32)
    tab = np.zeros(4, dtype=np.int32)
    assert lib.dr_plan_varlen(ok.ctypes.data, 1, 64, tab.ctypes.data, None, 2, ctypes.byref(n)) == B.DR_ERR_INVALID_ARG
    assert n.value == 4


def test_decode_rejects_bad_arguments_before_launch(lib):
    """dr_decode validates on the host: NULL state, packed layout, sizes outside
    {16, 32, 64, 128}, misaligned pointers."""
    d = desc(T=1)
    p16 = 16
    call = lambda dd, state=p16, q=p16: lib.dr_decode(ctypes.byref(dd), q, p16, p16, p16, p16,
                                                        state, p16, None)
    assert call(d, state=None) == B.DR_ERR_INVALID_ARG
    assert call(desc(T=1, d_k=96)) == B.DR_ERR_UNSUPPORTED
    assert call(desc(T=1, num_seqs=3)) == B.DR_ERR_INVALID_ARG
    assert call(d, q=18) == B.DR_ERR_ALIGNMENT
    dn = desc(T=1, variant=B.DR_DELTANET)
    assert call(dn) == B.DR_ERR_INVALID_ARG  # a gate pointer for DeltaNet


def test_prepare_flag_host_rules(lib):
    """DR_FLAG_PREPARE_INPUTS: accepted by dr_workspace_bytes; the bf16 tensor-core
    path prepares on the fly and keeps only the two inverse row norms per token and
    head (fp32, 512 bytes per chunk record), the fp32 CUDA-core path adds room for the
    prepared tensors (two q/k-sized buffers in the io dtype plus fp32 beta and gate);
    refused by dr_fwd_noalloc; an unknown flag bit stays an error."""
    n = B.DR_FLAG_PREPARE_INPUTS
    for kw in (dict(), dict(variant=B.DR_KDA)):
        d = desc(**kw)
        recs = (d.T + 63) // 64 * d.B * d.H
        extra = B.workspace_bytes(desc(flags=n, **kw)) - B.workspace_bytes(d)
        assert recs * 512 <= extra <= recs * 512 + 1023
    for kw, gate_per_token in ((dict(io_dtype=B.DR_F32, d_k=32, d_v=32, chunk=16), 1),
                               (dict(io_dtype=B.DR_F32, d_k=32, d_v=32, chunk=16,
                                     variant=B.DR_KDA), 128),
                               (dict(io_dtype=B.DR_F32, d_k=32, d_v=32, chunk=16,
                                     variant=B.DR_DELTANET), 0)):
        base = B.workspace_bytes(desc(**kw))
        prep = B.workspace_bytes(desc(flags=n, **kw))
        d = desc(**kw)
        th = d.B * d.T * d.H
        esize = 2 if d.io_dtype == B.DR_BF16 else 4
        need = 2 * th * d.d_k * esize + th * 4 + th * (d.d_k if gate_per_token == 128 else
                                                       gate_per_token) * 4
        assert esize == 4
        assert need <= prep - base <= need + 4 * 256 + 255
    assert call_fwd(desc(flags=n | 4)) == B.DR_ERR_INVALID_ARG
    d = desc(io_dtype=B.DR_F32, d_k=32, d_v=32, chunk=16, flags=n)
    assert lib.dr_fwd_noalloc(ctypes.byref(d), 16, 16, 16, 16, 16, None, 16, None,
                              None) == B.DR_ERR_UNSUPPORTED
    # on the fp32 path a workspace sized without the flag is too small with it
    f32 = dict(io_dtype=B.DR_F32, d_k=32, d_v=32, chunk=16)
    small = B.workspace_bytes(desc(**f32))
    assert call_fwd(desc(flags=n, **f32), ws_bytes=small) == B.DR_ERR_WORKSPACE
    dd = desc(T=1, flags=8)
    assert lib.dr_decode(ctypes.byref(dd), 16, 16, 16, 16, 16, 16, 16, None) == B.DR_ERR_INVALID_ARG


def test_gdn2_host_rules(lib):
    """Gated DeltaNet-2 has its own entry points: dr_fwd / dr_bwd refuse the variant,
    dr_gdn2_* refuse the others; sizes outside {16, 32, 64} and the preparation flag
    are unsupported; its workspace is sized by dr_workspace_bytes."""
    d2 = dict(variant=B.DR_GDN2, d_k=64, d_v=32, chunk=32)
    assert B.workspace_bytes(desc(**d2)) > 0
    assert B.workspace_bytes(desc(variant=B.DR_GDN2)) == 0            # d = 128
    assert call_fwd(desc(**d2)) == B.DR_ERR_INVALID_ARG

    def fwd2(d, **kw):
        p = dict(q=16, k=16, v=16, erase=16, write=16, g=16, h0=None, o=16, hT=None)
        p.update(kw)
        return B.dr_gdn2_fwd(d, *p.values(), 16, 1 << 40, None)
    assert fwd2(desc()) == B.DR_ERR_INVALID_ARG                       # variant GDN
    assert fwd2(desc(variant=B.DR_GDN2)) == B.DR_ERR_UNSUPPORTED
    assert fwd2(desc(flags=B.DR_FLAG_PREPARE_INPUTS, **d2)) == B.DR_ERR_UNSUPPORTED
    assert fwd2(desc(**d2), erase=None) == B.DR_ERR_INVALID_ARG
    assert fwd2(desc(**d2), g=None) == B.DR_ERR_INVALID_ARG
    assert fwd2(desc(**d2), write=8) == B.DR_ERR_ALIGNMENT
    assert B.dr_gdn2_fwd(desc(**d2), 16, 16, 16, 16, 16, 16, None, 16, None, 16, 100,
                         None) == B.DR_ERR_WORKSPACE

    def bwd2(d, **kw):
        p = dict(q=16, k=16, v=16, erase=16, write=16, g=16, h0=None, dO=16, dhT=None, dq=16,
                 dk=16, dv=16, derase=16, dwrite=16, dg=16, dh0=None)
        p.update(kw)
        return B.dr_gdn2_bwd(d, *p.values(), 16, 1 << 40, None)
    assert bwd2(desc(**d2), dwrite=None) == B.DR_ERR_INVALID_ARG
    assert bwd2(desc(**d2), dh0=4) == B.DR_ERR_ALIGNMENT
    assert bwd2(desc(variant=B.DR_KDA, d_k=64, d_v=64)) == B.DR_ERR_INVALID_ARG


def test_selftest_wait_rejects_bad_arguments_before_launch(lib):
    assert B.selftest_wait(None, False, 1000, None) == B.DR_ERR_INVALID_ARG
    assert B.selftest_wait(24, False, 1000, None) == B.DR_ERR_INVALID_ARG      # misaligned
    assert B.selftest_wait(16, False, -1, None) == B.DR_ERR_INVALID_ARG
    assert B.selftest_wait(16, True, 10 ** 9, None) == B.DR_ERR_INVALID_ARG   # > 100 ms


def test_gdn2_decode_host_rules(lib):
    p16 = 16

    def call(dd, **kw):
        a = dict(q=p16, k=p16, v=p16, erase=p16, write=p16, g=p16, state=p16, o=p16)
        a.update(kw)
        return lib.dr_gdn2_decode(ctypes.byref(dd), *a.values(), None)
    d2 = desc(T=1, variant=B.DR_GDN2)
    assert call(desc(T=1)) == B.DR_ERR_INVALID_ARG                    # not DR_GDN2
    assert call(d2, erase=None) == B.DR_ERR_INVALID_ARG
    assert call(d2, state=None) == B.DR_ERR_INVALID_ARG
    assert call(d2, write=8) == B.DR_ERR_ALIGNMENT
    assert call(desc(T=1, variant=B.DR_GDN2, d_k=96)) == B.DR_ERR_UNSUPPORTED
    assert call(desc(T=1, variant=B.DR_GDN2, flags=B.DR_FLAG_PREPARE_INPUTS)) == B.DR_ERR_UNSUPPORTED
    # dr_decode itself refuses the variant (its beta has no place in it)
    assert lib.dr_decode(ctypes.byref(d2), p16, p16, p16, p16, p16, p16, p16, None) == B.DR_ERR_INVALID_ARG
