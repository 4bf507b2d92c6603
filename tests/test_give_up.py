"""The give-up path of the kernels' bounded waits, on the GPU, without a
fault.  Every wait inside a kernel has an iteration limit; when one runs
out, the kernel issues nothing more, lets what it already issued complete,
writes nothing more, reports bit 4 of dev_status for the (sequence, v-head)
pairs it did not finish and returns (the home-server page's lesson on GDN
state faults: report the failure, never leave it silent).

GDN_FLAG_TEST_STALL makes the streaming recurrent kernel and the prefill's
chain role (the chunk-to-chunk recurrence) first wait on a barrier that nothing arrives on; that wait gives
up after a few microseconds.  The tests check the report, that no state or
output byte changed, and that the same context then runs a normal call that
matches the oracle (the context stayed usable)."""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_decode_gb300 as gdn
import gdn_inputs
import oracle
from tests import gpu_util as G

pytestmark = pytest.mark.gpu
BIT_GAVE_UP = 16


def _decode_call(c, stall, conv, S, out, st):
    d = gdn.make_dims(c.Hk, c.Hv, c.act_dtype, torch.float32, test_stall=stall)
    gdn.gdn_decode_step(d, G.weights(c), G.dev(c.x), G.dev(c.z), G.dev(c.a_raw), G.dev(c.b_raw), conv, S, out,
                        None, st)


def test_decode_wait_gives_up_and_reports():
    """Decode B=64 (16/32), the streaming kernel's shape."""
    c = gdn_inputs.decode_b64()
    conv, S = G.dev(c.conv0), G.dev(c.S0)
    conv0, S0 = conv.clone(), S.clone()
    out = torch.full((c.N, c.Hv * 128), 7.0, device="cuda")
    st = torch.zeros(c.N * c.Hv, device="cuda", dtype=torch.int32)
    _decode_call(c, True, conv, S, out, st)
    torch.cuda.synchronize()
    assert torch.all(st == BIT_GAVE_UP), st.unique()
    assert torch.equal(S, S0) and torch.equal(conv, conv0)
    assert torch.all(out == 7.0)
    # the context is usable: a normal step on the same buffers matches the oracle
    st.zero_()
    _decode_call(c, False, conv, S, out, st)
    torch.cuda.synchronize()
    ref = oracle.forward(c.Hk, c.Hv, c.x, c.z, c.a_raw, c.b_raw, c.conv_w, c.dt_bias, c.ssm_a, c.norm_w, c.conv0,
                         c.S0, cu_seqlens=np.arange(c.N + 1))
    assert torch.count_nonzero(st) == 0
    G.assert_out_close(out, ref.out, c.act_dtype)
    G.assert_state_close(S, ref.S, c.act_dtype)


def test_verify_wait_gives_up_and_reports():
    """Verify B=64, K=3 (16/32): no checkpoint or output is written."""
    c = gdn_inputs.verify_b64_k3()
    B, K = c.N, c.K
    d = gdn.make_dims(c.Hk, c.Hv, c.act_dtype, torch.float32, test_stall=True)
    ck_conv = torch.full((B, K, 3, c.C), 3.0, device="cuda", dtype=c.act_dtype)
    ck_S = torch.full((B, K, c.Hv, 128, 128), 5.0, device="cuda")
    out = torch.full((B * K, c.Hv * 128), 7.0, device="cuda")
    st = torch.zeros(B * c.Hv, device="cuda", dtype=torch.int32)
    gdn.gdn_verify_k(d, G.weights(c), K, G.dev(c.x), G.dev(c.z), G.dev(c.a_raw), G.dev(c.b_raw), G.dev(c.conv0),
                     G.dev(c.S0), ck_conv, ck_S, out, None, st)
    torch.cuda.synchronize()
    assert torch.all(st == BIT_GAVE_UP)
    assert torch.all(ck_S == 5.0) and torch.all(ck_conv == 3.0) and torch.all(out == 7.0)


def test_prefill_wait_gives_up_and_reports():
    """Tensor-core prefill (bf16), two sequences with a nonzero initial state."""
    c = gdn_inputs.make_case("stall", Hk=2, Hv=4, lengths=[100, 70], seed=4501)
    cu = c.cu_seqlens.to(torch.int32).contiguous()
    conv, S = G.dev(c.conv0), G.dev(c.S0)
    conv0, S0 = conv.clone(), S.clone()
    out = torch.full((c.T, c.Hv * 128), 7.0, device="cuda")
    st = torch.zeros(c.N * c.Hv, device="cuda", dtype=torch.int32)

    def call(stall):
        d = gdn.make_dims(c.Hk, c.Hv, c.act_dtype, torch.float32, test_stall=stall)
        nws = gdn.gdn_prefill_workspace_bytes(d, c.N, c.T)
        ws = torch.empty(max(nws, 16), device="cuda", dtype=torch.uint8)
        gdn.gdn_prefill_chunked(d, G.weights(c), cu, G.dev(cu), G.dev(c.x), G.dev(c.z), G.dev(c.a_raw),
                                G.dev(c.b_raw), conv, S, out, workspace=ws, dev_status=st)
        torch.cuda.synchronize()

    call(True)
    assert torch.all(st == BIT_GAVE_UP), st
    assert torch.equal(S, S0) and torch.equal(conv, conv0)
    assert torch.all(out == 7.0)
    st.zero_()
    call(False)
    ref = oracle.forward(c.Hk, c.Hv, c.x, c.z, c.a_raw, c.b_raw, c.conv_w, c.dt_bias, c.ssm_a, c.norm_w, c.conv0,
                         c.S0, cu_seqlens=cu.numpy())
    assert torch.count_nonzero(st) == 0
    G.assert_out_close(out, ref.out, c.act_dtype)
    G.assert_state_close(S, ref.S, c.act_dtype)


def test_projection_wait_gives_up_and_reports():
    """The weight-streaming projection kernel (gdn_in_proj at the B=64 decode batch, 35B dims):
    the status word reports bit 4, no output is written, and a normal
    call in the same context then matches the oracle."""
    T, H, Hk, Hv = 64, 2048, 16, 32
    c = gdn_inputs.make_proj_case(T=T, H=H, Hk=Hk, Hv=Hv, seed=4511)
    dv = lambda t: t.cuda().contiguous()
    bf = dict(device="cuda", dtype=torch.bfloat16)
    outs = [torch.full((T, 128 * (2 * Hk + Hv)), 7.0, **bf), torch.full((T, 128 * Hv), 7.0, **bf),
            torch.full((T, Hv), 7.0, **bf), torch.full((T, Hv), 7.0, **bf)]
    st = torch.zeros(1, device="cuda", dtype=torch.int32)
    ins = [dv(c.hidden), dv(c.W_qkv), dv(c.W_z), dv(c.W_a), dv(c.W_b)]

    def call(stall):
        d = gdn.make_dims(Hk, Hv, torch.bfloat16, torch.bfloat16, test_stall=stall)
        gdn.gdn_in_proj(d, *ins, *outs, dev_status=st)
        torch.cuda.synchronize()

    call(True)
    assert int(st.item()) == BIT_GAVE_UP
    assert all(torch.all(o == 7.0) for o in outs)
    st.zero_()
    call(False)
    assert int(st.item()) == 0
    refs = oracle.in_proj(c.hidden, c.W_qkv, c.W_z, c.W_a, c.W_b)
    for got, ref in zip(outs, refs):
        err = np.abs(got.float().cpu().numpy().astype(np.float64) - ref)
        assert np.all(err <= G.half_ulp_bf16(ref) + 1e-4)


def test_decode_with_folded_projections_gives_up_and_reports():
    """gdn_decode_step_ab at B=64 (the streaming kernel with the ssm_alpha / ssm_beta operands
    in its stages): every (sequence, v-head) reports bit 4 and nothing is written."""
    c = gdn_inputs.decode_b64()
    pc = gdn_inputs.make_proj_case(T=c.N, H=2048, Hk=c.Hk, Hv=c.Hv, seed=4512)
    d = gdn.make_dims(c.Hk, c.Hv, c.act_dtype, torch.float32, test_stall=True)
    conv, S = G.dev(c.conv0), G.dev(c.S0)
    conv0, S0 = conv.clone(), S.clone()
    out = torch.full((c.N, c.Hv * 128), 7.0, device="cuda")
    st = torch.zeros(c.N * c.Hv, device="cuda", dtype=torch.int32)
    gdn.gdn_decode_step_ab(d, G.weights(c), G.dev(c.x), G.dev(c.z), G.dev(pc.hidden), G.dev(pc.W_a), G.dev(pc.W_b),
                           conv, S, out, dev_status=st)
    torch.cuda.synchronize()
    assert torch.all(st == BIT_GAVE_UP), st.unique()
    assert torch.equal(S, S0) and torch.equal(conv, conv0)
    assert torch.all(out == 7.0)
