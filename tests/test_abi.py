"""The C-ABI library builds, loads and exports every entry point that
include/gdn.h and include/gdn_proj.h declare, and its host-side validation rejects bad arguments
before anything reaches a device (CPU only: no call here launches a kernel)."""
import ctypes
import os
import re
import subprocess

import pytest

import gated_deltanet_linear_decode_gb300 as gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")
HEADERS = [os.path.join(ROOT, "include", f) for f in ("gdn.h", "gdn_proj.h")]


def declared_functions():
    src = "".join(open(h).read() for h in HEADERS)
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("gdn_conv_state_init", "gdn_decode_step", "gdn_prefill_chunked", "gdn_verify_k",
                     "gdn_commit", "gdn_status_string", "gdn_prefill_workspace_bytes"):
        assert required in names


def test_library_exports_every_declared_symbol():
    lib_path = gdn._build.build()
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True, check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    lib = gdn.library()
    for n in declared_functions():
        assert hasattr(lib, n)
    assert set(gdn.EXPORTED_SYMBOLS) <= set(declared_functions())


def test_header_compiles_as_c():
    """The header is plain C (no CUDA or C++ types needed)."""
    src = ('#include "gdn.h"\n#include "gdn_proj.h"\n'
           'int main(void){ gdn_dims d; gdn_in_proj_weights w; (void)d; (void)w; return (int)GDN_OK; }\n')
    r = subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-fsyntax-only", "-I", os.path.dirname(HEADER),
                        "-x", "c", "-"], input=src, text=True, capture_output=True)
    assert r.returncode == 0, r.stderr


def test_status_strings_and_version():
    assert gdn.gdn_status_string(0) == "ok"
    assert "align" in gdn.gdn_status_string(3)
    assert gdn.gdn_status_string(99) == "unknown status"
    assert gdn.gdn_version() >= 100


# --- validation paths: every one returns before any CUDA call -------------------------------
FAKE = 0x10000          # a 16-byte aligned non-null address; never dereferenced on these paths


def _call(fn, *args):
    return getattr(gdn.library(), fn)(*args)


def _dims(Hk=16, Hv=32, act=1, out=0, eps=1e-6, flags=0):
    return gdn.GdnDims(Hk, Hv, eps, act, out, flags)


def _w(ptr=FAKE):
    return gdn.GdnWeights(ptr, ptr + 0x100000, ptr + 0x200000, ptr + 0x300000)


def _decode(d, w, B=4, x=FAKE, **kw):
    args = dict(z=FAKE + 0x1000000, a=FAKE + 0x2000000, b=FAKE + 0x3000000, cs=FAKE + 0x4000000,
                S=FAKE + 0x5000000, out=FAKE + 0x6000000, pre=None, st=None)
    args.update(kw)
    return _call("gdn_decode_step", ctypes.byref(d), ctypes.byref(w) if w is not None else None, B, x,
                 args["z"], args["a"], args["b"], args["cs"], args["S"], args["out"], args["pre"], args["st"], None)


@pytest.mark.parametrize("dims,status", [
    (None, 1),
    (_dims(Hk=0), 1), (_dims(Hv=0), 1), (_dims(Hk=16, Hv=40), 1),   # H_v % H_k != 0
    (_dims(eps=0.0), 1), (_dims(eps=float("nan")), 1), (_dims(act=7), 1), (_dims(out=-1), 1),
    (_dims(flags=0x80), 1), (_dims(flags=8), 1), (_dims(Hk=1, Hv=17), 2),                 # ratio > 16: unsupported
    (_dims(act=0, flags=4), 2),                                                           # bf16 state, fp32 activations
])
def test_decode_rejects_bad_dims(dims, status):
    if dims is None:
        st = _call("gdn_decode_step", None, ctypes.byref(_w()), 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                   None, None, None)
    else:
        st = _decode(dims, _w())
    assert st == status


def test_decode_validation():
    d = _dims()
    assert _decode(d, _w(), B=-1) == 1
    assert _decode(d, _w(), B=0) == 0                 # no-op
    assert _decode(d, None) == 1                      # no weights
    assert _decode(d, _w(), x=None) == 1              # null input
    assert _decode(d, _w(), x=FAKE + 8) == 3          # misaligned
    assert _decode(d, _w(FAKE + 4)) == 3              # misaligned weights
    assert _decode(d, _w(), out=FAKE) == 1            # output overlaps x
    assert _decode(d, _w(), pre=FAKE + 0x6000000) == 1   # prenorm overlaps out


def _decode_ab(d, w, B=4, H=2048, hidden=FAKE + 0x2000000, **kw):
    args = dict(z=FAKE + 0x1000000, Wa=FAKE + 0x7000000, Wb=FAKE + 0x8000000, cs=FAKE + 0x4000000,
                S=FAKE + 0x5000000, out=FAKE + 0x6000000, pre=None, st=None)
    args.update(kw)
    return _call("gdn_decode_step_ab", ctypes.byref(d), ctypes.byref(w) if w is not None else None, B, H, FAKE,
                 args["z"], hidden, args["Wa"], args["Wb"], args["cs"], args["S"], args["out"], args["pre"],
                 args["st"], None)


def test_decode_ab_validation():
    """The decode step with ssm_alpha / ssm_beta folded in: H, the activation type, the three
    projection pointers and their overlaps are checked before any CUDA call."""
    d = _dims()
    assert _decode_ab(d, _w(), B=0) == 0              # no-op
    assert _decode_ab(d, _w(), H=0) == 1
    assert _decode_ab(d, _w(), H=2044) == 1           # H not a multiple of 8
    assert _decode_ab(_dims(act=0), _w()) == 2        # fp32 activations
    assert _decode_ab(d, _w(), hidden=None) == 1
    assert _decode_ab(d, _w(), Wa=None) == 1
    assert _decode_ab(d, _w(), Wb=FAKE + 0x8000000 + 8) == 3
    assert _decode_ab(d, _w(), out=FAKE + 0x2000000) == 1   # output overlaps hidden
    assert _decode_ab(d, _w(), S=FAKE + 0x7000000) == 1     # state overlaps W_a


def test_verify_and_commit_validation():
    d = _dims()
    w = _w()
    L = gdn.library()
    base = [FAKE * (i + 1) * 0x100 for i in range(12)]
    # K out of range
    for K in (0, 17):
        assert L.gdn_verify_k(ctypes.byref(d), ctypes.byref(w), 2, K, *base[:10], None, None) == 1
    # S_ckpt overlapping S
    args = base[:10]
    args[7] = args[5]
    assert L.gdn_verify_k(ctypes.byref(d), ctypes.byref(w), 2, 3, *args, None, None) == 1
    assert L.gdn_commit(ctypes.byref(d), 2, 0, *base[:5], None) == 1
    assert L.gdn_commit(ctypes.byref(d), 0, 3, *base[:5], None) == 0
    assert L.gdn_commit(ctypes.byref(d), 2, 3, base[0], base[1], base[2], base[3] + 4, base[4], None) == 3


def test_ring_validation():
    d = _dims()
    w = _w()
    L = gdn.library()
    base = [FAKE * (i + 1) * 0x100 for i in range(12)]
    # verify: B, K, R, x, z, a, b, conv_state, S_ring, ring_cur, conv_ckpt, out, prenorm, status, stream
    ok = L.gdn_verify_k_ring(ctypes.byref(d), ctypes.byref(w), 0, 3, 4, *base[:9], None, None, None)
    assert ok == 0                                                    # B = 0: no-op
    for R in (3, 18):                                                 # R < K + 1, R > 17
        assert L.gdn_verify_k_ring(ctypes.byref(d), ctypes.byref(w), 2, 3, R, *base[:9], None, None, None) == 1
    args = base[:9]
    args[6] = None                                                    # no ring_cur
    assert L.gdn_verify_k_ring(ctypes.byref(d), ctypes.byref(w), 2, 3, 4, *args, None, None, None) == 1
    args = base[:9]
    args[7] = args[5]                                                 # conv_ckpt on S_ring
    assert L.gdn_verify_k_ring(ctypes.byref(d), ctypes.byref(w), 2, 3, 4, *args, None, None, None) == 1
    # commit: B, K, R, accept_len, conv_ckpt, conv_state, ring_cur
    assert L.gdn_commit_ring(ctypes.byref(d), 2, 3, 3, *base[:4], None) == 1          # R < K + 1
    assert L.gdn_commit_ring(ctypes.byref(d), 2, 3, 4, base[0], base[1], base[2], None, None) == 1
    assert L.gdn_commit_ring(ctypes.byref(d), 2, 3, 4, base[0], base[1], base[1], base[3], None) == 1
    assert L.gdn_commit_ring(ctypes.byref(d), 0, 3, 4, *base[:4], None) == 0
    # decode: B, R, x, z, a, b, conv_state, S_ring, ring_cur, out, prenorm, status, stream
    assert L.gdn_decode_step_ring(ctypes.byref(d), ctypes.byref(w), 2, 0, *base[:8], None, None, None) == 1
    args = base[:8]
    args[6] = None
    assert L.gdn_decode_step_ring(ctypes.byref(d), ctypes.byref(w), 2, 2, *args, None, None, None) == 1


def test_guard_validation():
    d = _dims()
    L = gdn.library()
    a, b, c = FAKE * 0x100, FAKE * 0x200, FAKE * 0x300
    assert L.gdn_state_faults(ctypes.byref(d), -1, a, 4, b, None) == 1
    assert L.gdn_state_faults(ctypes.byref(d), 2, a, -1, b, None) == 1
    assert L.gdn_state_faults(ctypes.byref(d), 2, None, 4, b, None) == 1
    assert L.gdn_state_faults(ctypes.byref(d), 2, a, 4, a + 16, None) == 1          # report overlaps the words
    assert L.gdn_state_faults(ctypes.byref(d), 2, a, 4, b + 4, None) == 3
    # reset: N, R, S, ring_cur, conv_state, dev_status
    assert L.gdn_state_reset(ctypes.byref(d), 2, 2, a, None, None, b, None) == 1     # R without ring_cur
    assert L.gdn_state_reset(ctypes.byref(d), 2, 0, a, c, None, b, None) == 1        # ring_cur without R
    assert L.gdn_state_reset(ctypes.byref(d), 2, 18, a, c, None, b, None) == 1
    assert L.gdn_state_reset(ctypes.byref(d), 0, 0, a, None, None, b, None) == 0     # no-op
    assert L.gdn_state_reset(ctypes.byref(d), 2, 0, a, None, None, a + 64, None) == 1   # status inside S
    assert L.gdn_state_reset(ctypes.byref(d), 2, 0, None, None, None, b, None) == 1


def test_projection_validation():
    L = gdn.library()
    d = _dims()                                    # bf16 activations, fp32 out
    d_bf = _dims(out=1)
    w = gdn.GdnInProjWeights(FAKE * 0x100, FAKE * 0x200, FAKE * 0x300, FAKE * 0x400)
    outs = [FAKE * 0x500, FAKE * 0x600, FAKE * 0x700, FAKE * 0x800]
    call = lambda dims, T, H, hid, ww, o=outs, ws=None, nws=0, st=None: L.gdn_in_proj(
        ctypes.byref(dims), T, H, hid, ctypes.byref(ww) if ww is not None else None, *o, ws, nws, st, None)
    assert call(d, 4, 2048, FAKE * 0x900, w) == 2                  # fp32 output type: unsupported
    assert call(_dims(act=0, out=1), 4, 2048, FAKE * 0x900, w) == 2
    assert call(d_bf, 0, 2048, FAKE * 0x900, w) == 0                # T = 0: no-op
    assert call(d_bf, -1, 2048, FAKE * 0x900, w) == 1
    assert call(d_bf, 4, 2047, FAKE * 0x900, w) == 1                # H not a multiple of 8
    assert call(d_bf, 4, 2048, None, w) == 1
    assert call(d_bf, 4, 2048, FAKE * 0x900, None) == 1
    assert call(d_bf, 4, 2048, FAKE * 0x900 + 8, w) == 3
    assert call(d_bf, 4, 2048, FAKE * 0x900, w, ws=None, nws=64) == 1   # workspace size without a workspace
    assert call(d_bf, 4, 2048, outs[0], w) == 1                     # hidden overlaps x
    assert call(d_bf, 4, 2048, FAKE * 0x900, w, st=FAKE * 0xa00 + 2) == 3   # status word off 4 bytes
    assert call(d_bf, 4, 2048, FAKE * 0x900, w, st=outs[1]) == 1    # status word inside z
    op = lambda dims, y, o, st=None: L.gdn_out_proj(ctypes.byref(dims), 4, 2048, y, FAKE * 0x200, o, None, 0, st, None)
    assert op(d_bf, FAKE * 0x100, FAKE * 0x100) == 1
    assert op(d_bf, FAKE * 0x100, FAKE * 0x300 + 4) == 3
    assert op(d, FAKE * 0x100, FAKE * 0x300) == 2
    assert op(d_bf, FAKE * 0x100, FAKE * 0x300, st=FAKE * 0x300) == 1   # status word inside out


def test_prefill_validation():
    d = _dims(Hk=16, Hv=48)
    w = _w()
    L = gdn.library()
    P = [FAKE * (i + 1) * 0x1000 for i in range(12)]

    def call(cu, n=None, **kw):
        arr = (ctypes.c_int32 * len(cu))(*cu)
        n = len(cu) - 1 if n is None else n
        a = dict(cu_dev=P[0], x=P[1], z=P[2], a=P[3], b=P[4], cs=P[5], S=P[6], out=P[7])
        a.update(kw)
        return L.gdn_prefill_chunked(ctypes.byref(d), ctypes.byref(w), n, arr, a["cu_dev"], a["x"], a["z"], a["a"],
                                     a["b"], a["cs"], a["S"], 0, a["out"], None, None, 0, None, None)
    assert call([0, 5], n=-1) == 1
    assert call([0, 5], n=0) == 0
    assert call([1, 5]) == 1                 # must start at 0
    assert call([0, 5, 3]) == 1              # decreasing
    assert call([0, 5], x=None) == 1
    assert call([0, 5], x=P[1] + 2) == 3
    assert call([0, 5], cu_dev=None) == 1
    assert gdn.gdn_prefill_workspace_bytes(d, 1, 8192) >= 0
