"""gdn_prefill_chunked_static: the prefill entry point that allocates nothing.

Some callers cannot allocate device memory where they run the prefill -- a
serving runtime whose allocator owns the whole device pool, or a plugin that is
handed only its input and output buffers -- so they cannot supply the workspace
that gdn_prefill_chunked needs.  For them the library keeps one fixed scratch
area in device memory (GDN_PREFILL_STATIC_SCRATCH_BYTES, shared by every call).

Checked here through the C ABI: two calls of the static entry point in a row
(the second finds the first one's leftovers in the shared area) give the
results of gdn_prefill_chunked with a caller-provided workspace, within the
tolerances of the other GPU tests (tests/gpu_util.py); and a problem too large
for the area is refused on the host, before anything reaches a device.

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
    """Two ragged multi-sequence prefills with the model's head counts (16/48,
    bf16 in, fp32 out), run back to back through the static entry point, then
    through gdn_prefill_chunked with a torch-allocated workspace: outputs,
    pre-norm outputs and states agree within the bf16 tolerances, conv states
    bit for bit."""
    cases = [gdn_inputs.make_case("static_a", Hk=16, Hv=48, lengths=[300, 0, 333, 91], seed=2101),
             gdn_inputs.make_case("static_b", Hk=16, Hv=48, lengths=[17, 640], seed=2102)]
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
        tol_y, tol_s = G.TOL[torch.bfloat16]
        assert (g["out"] - ref["out"]).abs().max().item() <= tol_y
        assert (g["prenorm_out"] - ref["prenorm_out"]).abs().max().item() <= tol_y
        rel = ((g["S"] - ref["S"]).norm() / ref["S"].norm().clamp_min(1e-30)).item()
        assert rel <= tol_s, rel
        assert torch.equal(g["conv_state"].view(torch.int16), ref["conv_state"].view(torch.int16))
