"""gdn_prefill_chunked_static: the prefill entry point that allocates nothing.

Some callers cannot allocate device memory where they run the prefill -- a
serving runtime whose allocator owns the whole device pool, or a plugin that is
handed only its input and output buffers -- so they cannot supply the workspace
that gdn_prefill_chunked needs.  For them the library keeps one fixed scratch
area in device memory (GDN_PREFILL_STATIC_SCRATCH_BYTES, shared by every call).

Checked here through the C ABI: calls of the static entry point in a row
(each finds the previous one's leftovers in the shared area) give bit for
bit the results of gdn_prefill_chunked with a caller-provided workspace (the
same kernels on the same inputs); and a problem too large for the area is
refused on the host, before anything reaches a device.

This file is collected last so that a run stopping at its first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

import gated_deltanet_linear_decode_gb300 as gdn
import gdn_inputs
from tests import gpu_util as G

FAKE = 0x10000   # 16-byte aligned, non-null, never dereferenced on the refusal path
GDN_E_WORKSPACE = 5


def test_static_prefill_refuses_oversize_problem_on_the_host():
    """Beyond the area's size the call returns GDN_E_WORKSPACE without any CUDA
    call (CPU only); the size quoted in the header (1,280 tokens of one
    sequence with bf16 activations and 48 v-heads) is exactly the boundary."""
    lib = gdn.library()
    d = gdn.make_dims(16, 48, act_dtype=torch.bfloat16, out_dtype=torch.bfloat16)
    limit = gdn.PREFILL_STATIC_SCRATCH_BYTES
    assert gdn.gdn_prefill_workspace_bytes(d, 1, 1280) <= limit < gdn.gdn_prefill_workspace_bytes(d, 1, 1281)
    w = gdn.GdnWeights(FAKE, FAKE, FAKE, FAKE)
    for T in (1281, 1 << 16):
        cu = (ctypes.c_int32 * 2)(0, T)
        st = lib.gdn_prefill_chunked_static(ctypes.byref(d), ctypes.byref(w), 1, cu, FAKE, FAKE, FAKE, FAKE, FAKE,
                                            FAKE, FAKE, 1, FAKE, None, None, None)
        assert st == GDN_E_WORKSPACE, st
    assert "workspace" in gdn.gdn_status_string(GDN_E_WORKSPACE)


def _inputs(c):
    return dict(cu_seqlens_host=c.cu_seqlens.to(torch.int32).contiguous(),
                cu_seqlens_dev=G.dev(c.cu_seqlens.to(torch.int32)), x=G.dev(c.x), z=G.dev(c.z),
                a_raw=G.dev(c.a_raw), b_raw=G.dev(c.b_raw))


def _buffers(c):
    return dict(conv_state=G.dev(c.conv0), S=G.dev(c.S0),
                out=torch.empty(c.T, c.Hv * 128, device="cuda", dtype=torch.float32),
                prenorm_out=torch.empty(c.T, c.Hv * 128, device="cuda", dtype=torch.float32))


@pytest.mark.gpu
def test_static_prefill_matches_workspace_entry_point_on_two_calls():
    """Three prefills run back to back through the static entry point, then
    through gdn_prefill_chunked with a torch-allocated workspace: two ragged
    multi-sequence problems with the model's head counts (16/48, bf16 in, fp32
    out) and one long single sequence with few heads (2/4, 4,100 tokens, 65
    chunks, each v-head's chain walking them all).  Both entry points run the same deterministic kernels on the same
    inputs, so outputs, pre-norm outputs, states and conv states must agree
    bit for bit -- a stale byte read from the shared area (left by the call
    before) would show as a difference."""
    cases = [gdn_inputs.make_case("static_a", Hk=16, Hv=48, lengths=[300, 0, 333, 91], seed=2101),
             gdn_inputs.make_case("static_b", Hk=16, Hv=48, lengths=[17, 640], seed=2102),
             gdn_inputs.make_case("static_c", Hk=2, Hv=4, lengths=[4100], seed=2103)]
    for c in cases:
        d = G.dims(c, torch.float32)
        assert 0 < gdn.gdn_prefill_workspace_bytes(d, c.N, c.T) <= gdn.PREFILL_STATIC_SCRATCH_BYTES
    # two calls in a row of the entry point under test
    got = []
    for c in cases:
        d, w, inp, buf = G.dims(c, torch.float32), G.weights(c), _inputs(c), _buffers(c)
        gdn.gdn_prefill_chunked_static(d, w, **inp, **buf)
        got.append(buf)
    torch.cuda.synchronize()
    # the same problems through the workspace entry point
    for c, g in zip(cases, got):
        d, w, inp, ref = G.dims(c, torch.float32), G.weights(c), _inputs(c), _buffers(c)
        ws = torch.empty(gdn.gdn_prefill_workspace_bytes(d, c.N, c.T), device="cuda", dtype=torch.uint8)
        gdn.gdn_prefill_chunked(d, w, **inp, **ref, workspace=ws)
        torch.cuda.synchronize()
        for key in ("out", "prenorm_out", "S"):
            assert torch.equal(g[key].view(torch.int32), ref[key].view(torch.int32)), (c.name, key)
        assert torch.equal(g["conv_state"].view(torch.int16), ref["conv_state"].view(torch.int16))
