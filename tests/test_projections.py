"""GPU parity of the projections either side of the mixer (gdn_in_proj,
gdn_out_proj) against the fp64 oracle on the same bf16 inputs.  Each output
is one fp32 sum of exact bf16 products rounded once to bf16, so the bound is
half a bf16 ulp of the reference plus 1e-4 for the fp32 accumulation.

T <= 256 runs the library's weight-streaming kernel: a CTA per 128-row tile
when there are about as many tiles as SMs, else clusters of 2 or 4 CTAs that
split a tile's K and add their partial sums in distributed shared memory (both
are run: the input GEMMs take the first, ssm_out the second), with zero fill
past the last weight row and past the last multiple of 64 in K.  Larger T runs
cuBLASLt.  The status word of the streaming kernel must stay clear."""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_decode_gb300 as gdn
import gdn_inputs
import oracle
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def _close(got, ref):
    got = got.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    bound = G.half_ulp_bf16(ref) + 1e-4
    assert np.all(err <= bound), f"worst excess {float((err - bound).max()):.3e}"


def _run(c, T, rows=None, ws_bytes=0):
    d = gdn.make_dims(c.Hk, c.Hv, torch.bfloat16, torch.bfloat16)
    dv = lambda t: t.cuda().contiguous()
    C, HvD = 128 * (2 * c.Hk + c.Hv), 128 * c.Hv
    x = torch.empty(T, C, device="cuda", dtype=torch.bfloat16)
    z = torch.empty(T, HvD, device="cuda", dtype=torch.bfloat16)
    a = torch.empty(T, c.Hv, device="cuda", dtype=torch.bfloat16)
    b = torch.empty(T, c.Hv, device="cuda", dtype=torch.bfloat16)
    out = torch.empty(T, c.H, device="cuda", dtype=torch.bfloat16)
    ws = torch.empty(ws_bytes, device="cuda", dtype=torch.uint8) if ws_bytes else None
    st = torch.zeros(1, device="cuda", dtype=torch.int32)
    gdn.gdn_in_proj(d, dv(c.hidden), dv(c.W_qkv), dv(c.W_z), dv(c.W_a), dv(c.W_b), x, z, a, b, workspace=ws,
                    dev_status=st)
    gdn.gdn_out_proj(d, dv(c.y), dv(c.W_out), out, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    sel = slice(None) if rows is None else rows
    refs = oracle.in_proj(c.hidden[sel], c.W_qkv, c.W_z, c.W_a, c.W_b)
    for got, ref in zip((x, z, a, b), refs):
        _close(got[sel], ref)
    _close(out[sel], oracle.out_proj(c.y[sel], c.W_out))


@pytest.mark.parametrize("T,ws", [(300, 0), (257, 4 << 20), (256, 0), (192, 0), (129, 1 << 20), (64, 4 << 20),
                                  (64, 0), (48, 0), (17, 1 << 20), (1, 0)])
def test_projections_35b_dims(T, ws):
    """Hidden 2048, 16/32 heads: ragged prefills either side of the 256-row switch to cuBLASLt,
    the B=64 K=3 verify batch, the B=64 decode batch, 48 and 17 rows, and a single token, with
    and without a workspace."""
    c = gdn_inputs.make_proj_case(T=T, H=2048, Hk=16, Hv=32, seed=200 + T)
    _run(c, T, ws_bytes=ws)


def test_projections_27b_dims_full_size_sampled():
    """Hidden 5120, 16/48 heads, T = 8192 (the prefill workload): every output of 24 sampled rows."""
    T = 8192
    c = gdn_inputs.make_proj_case(T=T, H=5120, Hk=16, Hv=48, seed=210)
    rows = torch.randperm(T, generator=torch.Generator().manual_seed(3))[:24].sort().values
    _run(c, T, rows=rows, ws_bytes=32 << 20)


@pytest.mark.parametrize("T", [64, 192])
def test_projections_27b_dims_decode_batches(T):
    """Hidden 5120, 16/48 heads at the decode and verify batch sizes (130 tiles of input GEMMs, a
    CTA each; ssm_out's 40 tiles split two ways)."""
    c = gdn_inputs.make_proj_case(T=T, H=5120, Hk=16, Hv=48, seed=220 + T)
    _run(c, T)


@pytest.mark.parametrize("T", [5, 100])
def test_projections_ragged_hidden(T):
    """H = 2056: K ends 8 past a multiple of 64 (zero-filled copies), ssm_out's 2056 rows end 8
    into their last 128-row tile, and ssm_alpha / ssm_beta are 4-row GEMMs."""
    c = gdn_inputs.make_proj_case(T=T, H=2056, Hk=2, Hv=4, seed=230 + T)
    _run(c, T)
