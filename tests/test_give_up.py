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
