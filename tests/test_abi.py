"""The C ABI library loads, exports every declared entry point, and rejects
bad arguments on the host before any launch (no GPU needed).

Error contract (SANA `fused_gdn.py` page, `fused_gdn_func`): bad shapes,
dtypes and layouts are value errors; a reverse scan with state input/output
is "not implemented"."""
import ctypes
import os
import re

import pytest

import gated_delta_rule_18_gb300 as gdn
from gated_delta_rule_18_gb300 import TensorDesc
from gated_delta_rule_18_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")

OK, NULL, SHAPE, DTYPE, LAYOUT, UNSUP, CUDA, TIMEOUT, WS, DEVICE = range(10)
GDN_ACCUMULATE_FLAG = 0x1


@pytest.fixture(scope="module")
def L():
    build()
    return gdn.lib()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for s in ("gdn_prep", "gdn_chunk_fwd", "gdn_workspace_size", "gdn_status_string",
              "gdn_last_device_error"):
        assert s in syms


def test_every_declared_symbol_is_exported(L):
    for s in declared_symbols():
        assert hasattr(L, s), f"{s} declared in gdn.h but not exported"


def test_status_strings(L):
    for code in range(10):
        assert gdn.gdn_status_string(code)
    assert gdn.gdn_status_string(99) == "unknown status"


def test_workspace_size(L):
    f32 = gdn.gdn_workspace_size(1, 256, 2, 64, 64, 1, 0, gdn.F32, 0)
    b16 = gdn.gdn_workspace_size(4, 4096, 16, 128, 128, 4, 0, gdn.BF16, 0)
    assert 0 < f32 < b16
    # varlen adds the chunk table; the denominator widens u
    assert gdn.gdn_workspace_size(1, 4096, 16, 128, 128, 64, 1, gdn.BF16, 0) > \
        gdn.gdn_workspace_size(1, 4096, 16, 128, 128, 1, 0, gdn.BF16, 0)
    assert gdn.gdn_workspace_size(1, 4096, 16, 112, 112, 1, 0, gdn.BF16, 1) >= \
        gdn.gdn_workspace_size(1, 4096, 16, 112, 112, 1, 0, gdn.BF16, 0)
    # rejected shapes report 0
    assert gdn.gdn_workspace_size(1, 10, 1, 256, 64, 1, 0, gdn.BF16, 0) == 0   # K > 128
    assert gdn.gdn_workspace_size(2, 10, 1, 64, 64, 2, 1, gdn.BF16, 0) == 0    # varlen B != 1
    assert gdn.gdn_workspace_size(1, 10, 1, 64, 256, 1, 0, gdn.BF16, 1) == 0   # V + den > 256


# Fake, never-dereferenced, well-aligned device addresses: every call below
# must be rejected by host-side checks before anything touches them.
A = 1 << 20


def P(i):
    return ctypes.c_void_p(A * (i + 1))


def desc(dtype, B, T, H, D):
    return TensorDesc(dtype, 0, T * H * D, H * D, D)


def fwd(L, **kw):
    a = dict(q=P(0), k=P(1), qkd=desc(gdn.BF16, 1, 128, 2, 64), v=P(2),
             vd=desc(gdn.BF16, 1, 128, 2, 64), g=P(3), gk=None, beta=P(4), h0=None, cu=None,
             n_seq=1, out=P(5), od=desc(gdn.BF16, 1, 128, 2, 64), hf=None, den=None, B=1,
             T=128, H=2, K=64, V=64, chunk=64, reverse=0, flags=0, ws=P(6), wsb=1 << 30,
             stream=None)
    a.update(kw)
    return L.gdn_chunk_fwd(a["q"], a["k"], a["qkd"], a["v"], a["vd"], a["g"], a["gk"],
                           a["beta"], a["h0"], a["cu"], a["n_seq"], a["out"], a["od"],
                           a["hf"], a["den"], a["B"], a["T"], a["H"], a["K"], a["V"],
                           a["chunk"], a["reverse"], a["flags"], a["ws"], a["wsb"],
                           a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), NULL), (dict(beta=None), NULL), (dict(out=None), NULL),
    (dict(g=None), NULL),                       # neither gate
    (dict(gk=P(7)), UNSUP),                     # both gates
    (dict(ws=None), WS), (dict(wsb=1024), WS), (dict(ws=ctypes.c_void_p(A + 16)), WS),
    (dict(chunk=32), SHAPE), (dict(K=136), SHAPE), (dict(K=60), SHAPE), (dict(V=60), SHAPE),
    (dict(V=256, den=P(8)), SHAPE), (dict(H=0), SHAPE), (dict(T=-1), SHAPE),
    (dict(n_seq=2), SHAPE),                      # dense needs n_seq == B
    (dict(cu=P(9), B=2, n_seq=2), SHAPE),        # varlen needs B == 1
    (dict(cu=P(9), n_seq=0), SHAPE),
    (dict(qkd=desc(7, 1, 128, 2, 64)), DTYPE),
    (dict(qkd=desc(gdn.F32, 1, 128, 2, 64)), DTYPE),   # q/k and v dtypes differ
    (dict(q=ctypes.c_void_p(A + 2)), LAYOUT),
    (dict(qkd=TensorDesc(gdn.BF16, 0, 128 * 2 * 64, 2 * 64 + 4, 64)), LAYOUT),
    (dict(g=ctypes.c_void_p(A + 2)), LAYOUT),
    (dict(reverse=1, h0=P(10)), UNSUP), (dict(reverse=1, hf=P(10)), UNSUP),
    (dict(flags=0x80), UNSUP),
])
def test_chunk_fwd_rejects_on_host(L, kw, code):
    assert fwd(L, **kw) == code


def test_prep_rejects_on_host(L):
    d = desc(gdn.BF16, 1, 16, 2, 64)
    assert L.gdn_prep(None, d, P(1), d, 1, 16, 2, 64, 0, 1.0, 1e-6, None, None) == NULL
    assert L.gdn_prep(P(0), d, P(1), desc(gdn.F32, 1, 16, 2, 64), 1, 16, 2, 64, 0, 1.0,
                      1e-6, None, None) == DTYPE
    assert L.gdn_prep(P(0), d, P(1), d, 1, 16, 2, 60, 0, 1.0, 1e-6, None, None) == SHAPE
    assert L.gdn_prep(P(0), d, P(1), d, 1, 16, 2, 512, 0, 1.0, 1e-6, None, None) == SHAPE
    assert L.gdn_prep(P(0), d, P(1), d, 1, 16, 2, 64, 0x7, 1.0, 1e-6, None, None) == UNSUP
    assert L.gdn_prep(ctypes.c_void_p(A + 8), d, P(1), d, 1, 16, 2, 64, 0, 1.0, 1e-6, None,
                      None) == LAYOUT
    # zero tokens: nothing to do, nothing launched
    assert L.gdn_prep(P(0), d, P(1), d, 1, 0, 2, 64, 0, 1.0, 1e-6, None, None) == OK


def test_merge_rejects_on_host(L):
    d16, d32 = desc(gdn.BF16, 1, 16, 2, 64), desc(gdn.F32, 1, 16, 2, 64)
    m = lambda num=P(0), nd=d16, den=P(4), gate=None, gd=d16, out=P(1), od=d16, V=64, eps=1e-6, T=16: \
        L.gdn_merge(num, nd, den, gate, gd, out, od, 1, T, 2, V, eps, None)
    assert m(num=None) == NULL
    assert m(od=d32) == DTYPE                       # bf16 num, fp32 out: not offered
    assert m(gate=P(2), gd=d32) == DTYPE            # gate dtype differs from num
    assert m(V=60) == SHAPE                         # V not a multiple of 8 (bf16)
    assert m(eps=-1.0) == SHAPE
    assert m(num=ctypes.c_void_p(A + 8)) == LAYOUT  # misaligned rows
    assert m(den=ctypes.c_void_p(A + 2)) == LAYOUT
    assert m(T=0) == OK                             # nothing to do, nothing launched


def test_frame_fwd_rejects_on_host(L):
    d16, d32 = desc(gdn.BF16, 1, 256, 2, 64), desc(gdn.F32, 1, 256, 2, 64)

    def ff(q=P(0), qkd=d16, vd=d16, gf=P(3), h0=None, hf=None, den=None, T=256, frame=64,
           direction=0, flags=0, ws=P(9), wsb=1 << 30):
        return L.gdn_frame_fwd(q, P(1), qkd, P(2), vd, gf, P(4), h0, P(5), d16, hf, den, 1, T, 2,
                               64, 64, frame, direction, flags, ws, wsb, None)
    assert ff(q=None) == NULL
    assert ff(qkd=d32) == DTYPE                    # the frame path takes bf16 q / k / v
    assert ff(frame=96) == SHAPE                   # not a multiple of 64
    assert ff(frame=192) == SHAPE                  # does not divide T
    assert ff(direction=3) == UNSUP
    assert ff(direction=1, h0=P(6)) == UNSUP       # state I/O is forward only
    assert ff(flags=0x2) == UNSUP
    assert ff(q=ctypes.c_void_p(A + 8)) == LAYOUT
    assert ff(wsb=16) == WS
    assert ff(T=0) == OK                           # nothing to do, nothing launched
    assert gdn.gdn_frame_workspace_size(1, 256, 2, 64, 64, 64, True) > 0
    assert gdn.gdn_frame_workspace_size(1, 256, 2, 64, 64, 96, True) == 0


def test_seg_fwd_and_summary_reject_on_host(L):
    d16, d32 = desc(gdn.BF16, 1, 256, 2, 64), desc(gdn.F32, 1, 256, 2, 64)

    def sf(q=P(0), qkd=d16, vd=d16, seg=128, T=256, h0=None, reverse=0, flags=0, ws=P(9),
           wsb=1 << 30):
        return L.gdn_chunk_fwd_seg(q, P(1), qkd, P(2), vd, P(3), None, P(4), h0, P(5), d16,
                                   None, None, 1, T, 2, 64, 64, 64, reverse, flags, seg, ws, wsb,
                                   None)
    assert sf(q=None) == NULL
    assert sf(qkd=d32, vd=d32) == DTYPE            # fp32 runs the fused path only
    assert sf(seg=96) == SHAPE                     # not a multiple of 64
    assert sf(seg=0) == SHAPE
    assert sf(reverse=1, h0=P(6)) == UNSUP
    assert sf(wsb=1024) == WS
    need = gdn.gdn_seg_workspace_size(1, 256, 2, 64, 64, False, 128)
    assert need > gdn.gdn_workspace_size(1, 256, 2, 64, 64, 1, 0, gdn.BF16, 0)
    assert gdn.gdn_seg_workspace_size(1, 256, 2, 64, 64, False, 100) == 0

    def ss(k=P(0), kd=d16, ext=P(5), tr=P(6), seg=128, T=256, flags=0, wsb=1 << 30):
        return L.gdn_state_summary(k, kd, P(2), d16, P(3), None, P(4), ext, tr, 1, T, 2, 64, 64,
                                   64, seg, flags, P(9), wsb, None)
    assert ss(k=None) == NULL
    assert ss(ext=None) == NULL
    assert ss(kd=d32) == DTYPE
    assert ss(seg=32) == SHAPE
    assert ss(flags=GDN_ACCUMULATE_FLAG) == UNSUP  # summaries are stored, never added
    assert ss(ext=ctypes.c_void_p(A + 2)) == LAYOUT
    assert ss(wsb=16) == WS
    assert ss(T=0) == OK


def test_chunk_bwd_rejects_on_host(L):
    d16, d32 = desc(gdn.BF16, 1, 128, 2, 64), desc(gdn.F32, 1, 128, 2, 64)

    def bw(q=P(0), qkd=d16, vd=d16, dod=d16, gk=None, h0=None, dhf=None, dh0=P(16), dq=P(10), V=64,
           T=128, K=64, reverse=0, flags=0, wsb=1 << 30):
        return L.gdn_chunk_bwd(q, P(1), qkd, P(2), vd, P(3), gk, P(4), h0, None, 1, P(5), dod, None,
                               dhf, dq, P(11), P(12), P(13), P(14), dh0, 1, T, 2, K, V, 64, reverse,
                               flags, P(9), wsb, None)
    assert bw(dq=None) == NULL
    assert bw(qkd=d32) == DTYPE                # fp32 q / k with bf16 v
    assert bw(dod=d32) == DTYPE
    # the fp32 path (fp32 q, k, v and dout): its own shape and layout checks
    f32 = dict(qkd=d32, vd=d32, dod=d32)
    assert bw(vd=d16, dod=d32, qkd=d32) == DTYPE
    assert bw(dod=d16, qkd=d32, vd=d32) == DTYPE
    assert bw(K=129, **f32) == SHAPE           # K <= 128
    assert bw(V=264, **f32) == SHAPE
    assert bw(gk=P(7), **f32) == UNSUP
    assert bw(reverse=1, **f32) == UNSUP
    assert bw(dq=ctypes.c_void_p(A + 2), **f32) == LAYOUT   # 4-byte aligned fp32
    assert bw(wsb=1024, **f32) == WS
    assert bw(T=0, dh0=None, **f32) == OK      # nothing to do
    assert gdn.gdn_bwd_workspace_size(1, 256, 2, 64, 64, fp32=True) > 0
    assert gdn.gdn_bwd_workspace_size(1, 256, 2, 129, 64, fp32=True) == 0
    assert gdn.gdn_bwd_workspace_size(2, 256, 2, 64, 64, 3, True, fp32=True) == 0   # packed: B == 1
    # any V: ragged 16-column ranges, the ones column in the last
    assert gdn.gdn_bwd_workspace_size(1, 100, 2, 48, 40, with_den=True, fp32=True) > 0
    assert bw(V=264) == SHAPE                  # V <= 256
    assert bw(V=60) == SHAPE                   # a multiple of 8
    assert bw(gk=P(7)) == UNSUP                # g and gk both given
    assert bw(reverse=1) == UNSUP              # dh0 asked of a reverse scan
    assert bw(flags=GDN_ACCUMULATE_FLAG) == UNSUP
    assert bw(dq=ctypes.c_void_p(A + 4)) == LAYOUT
    assert bw(wsb=1024) == WS
    assert gdn.gdn_bwd_workspace_size(1, 128, 2, 64, 64) > gdn.gdn_workspace_size(
        1, 128, 2, 64, 64, 1, 0, gdn.BF16, 0)
    # V = 256 runs as two 128-column ranges over one range's workspace
    assert gdn.gdn_bwd_workspace_size(1, 128, 2, 64, 256) == gdn.gdn_bwd_workspace_size(1, 128, 2, 64, 128)
    assert gdn.gdn_bwd_workspace_size(1, 128, 2, 64, 264) == 0
    assert gdn.gdn_bwd_workspace_size(1, 300, 2, 64, 64, 3, True) > 0
    # the denominator's column: V = 128 runs as ranges of 120 and 8 + the ones column
    assert gdn.gdn_bwd_workspace_size(1, 128, 2, 64, 128, with_den=True) > 0


def test_bidir_rejects_on_host(L):
    d16, d32 = desc(gdn.BF16, 1, 128, 2, 64), desc(gdn.F32, 1, 128, 2, 64)

    def bd(g=P(3), gk=None, g_bwd=None, od=d16, flags=0, wsb=1 << 30, T=128):
        return L.gdn_chunk_fwd_bidir(P(0), P(1), d16, P(2), d16, g, gk, P(4), g_bwd, None, None, 1,
                                     P(5), od, P(6), 1, T, 2, 64, 64, 64, flags, P(9), wsb, None)
    assert bd(g=None, gk=P(7), g_bwd=P(8)) == UNSUP   # backward gates replace a scalar gate only
    assert bd(flags=GDN_ACCUMULATE_FLAG) == UNSUP      # out is overwritten
    assert bd(od=d32) == DTYPE                         # out in q's dtype
    assert bd(wsb=1024) == WS
    assert bd(T=0) == OK
    assert gdn.gdn_bidir_workspace_size(1, 128, 2, 64, 64, 1, 0, gdn.BF16, 1) > \
        2 * gdn.gdn_workspace_size(1, 128, 2, 64, 64, 1, 0, gdn.BF16, 1)


def test_seg_choose_sizes_the_grid():
    """Host arithmetic only: segments pay when few (sequence, head, value
    tile) CTAs would walk a long sequence, never when the plain pass already
    fills the SMs."""
    choose = gdn.gdn_seg_choose
    long_few = choose(1, 65536, 4, 128, 128, False, 152)
    assert 64 <= long_few < 65536 and long_few % 64 == 0
    assert choose(4, 4096, 16, 128, 128, False, 152) >= 4096    # 128 CTAs already
    assert choose(1, 256, 2, 64, 64, False, 152) >= 256         # four chunks
    assert choose(1, 65536, 4, 128, 128, False, 8) >= long_few  # fewer SMs, longer segments
    assert choose(1, 0, 4, 128, 128, False, 152) == 0
    assert choose(1, 64, 4, 128, 128, False, 0) == 0


def test_python_binding_fails_loudly_without_library(monkeypatch):
    monkeypatch.setattr(gdn, "_lib", None)
    monkeypatch.setattr(gdn, "LIB", "/nonexistent/libgdn.so")
    with pytest.raises(RuntimeError, match="not built"):
        gdn.lib()
