"""GPU parity of the decode step with the ssm_alpha / ssm_beta projections folded
into the recurrent kernels (gdn_decode_step_ab) against the fp64 oracle: the
oracle's in_proj forms a_raw = hidden . W_a^T and b_raw = hidden . W_b^T (xwen
CLAUDE.md page, "Architecture cheat sheet", "Gated DeltaNet layer"), unrounded
as the kernel keeps them, and its recurrence takes them from there.  Both
recurrent kernels are covered (the cluster kernel for small batches, the
streaming kernel at B = 64), with H a multiple of 64 and not, and with a bf16
state (the streaming kernel then holds each tile in shared memory; with the
folded operands one CTA per SM fits instead of two).  Tolerances:
tests/gpu_util.py."""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_decode_gb300 as gdn
import gdn_inputs
import oracle
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,Hk,Hv", [(1, 2048, 16, 32), (3, 2056, 2, 4), (64, 2048, 16, 32), (64, 5120, 16, 48)])
def test_decode_ab_matches_oracle(B, H, Hk, Hv):
    c = gdn_inputs.make_case("ab", Hk=Hk, Hv=Hv, B=B, K=1, seed=4600 + B + H)
    pc = gdn_inputs.make_proj_case(T=B, H=H, Hk=Hk, Hv=Hv, seed=4700 + B + H)
    d, w = G.dims(c, torch.float32), G.weights(c)
    conv, S = G.dev(c.conv0), G.dev(c.S0)
    out = torch.empty(B, Hv * 128, device="cuda", dtype=torch.float32)
    st = torch.zeros(B * Hv, device="cuda", dtype=torch.int32)
    gdn.gdn_decode_step_ab(d, w, G.dev(c.x), G.dev(c.z), G.dev(pc.hidden), G.dev(pc.W_a), G.dev(pc.W_b), conv, S,
                           out, dev_status=st)
    torch.cuda.synchronize()
    _, _, a64, b64 = oracle.in_proj(pc.hidden, pc.W_qkv, pc.W_z, pc.W_a, pc.W_b)
    ref = oracle.forward(Hk, Hv, c.x, c.z, a64, b64, c.conv_w, c.dt_bias, c.ssm_a, c.norm_w, c.conv0, c.S0,
                         cu_seqlens=np.arange(B + 1))
    G.assert_out_close(out, ref.out, c.act_dtype)
    G.assert_state_close(S, ref.S, c.act_dtype)
    assert G.conv_bits_equal(conv, ref.conv_state, c.act_dtype)
    assert int(st.abs().sum()) == 0


@pytest.mark.parametrize("B,H,Hk,Hv", [(64, 2048, 16, 32), (64, 5120, 16, 48), (2, 2048, 16, 32)])
def test_decode_ab_bf16_state_matches_oracle(B, H, Hk, Hv):
    c = gdn_inputs.make_case("abs", Hk=Hk, Hv=Hv, B=B, K=1, seed=4800 + B + H)
    pc = gdn_inputs.make_proj_case(T=B, H=H, Hk=Hk, Hv=Hv, seed=4900 + B + H)
    S0 = c.S0.to(torch.bfloat16)
    d, w = G.dims(c, torch.float32, state_dtype=torch.bfloat16), G.weights(c)
    conv, S = G.dev(c.conv0), G.dev(S0)
    out = torch.empty(B, Hv * 128, device="cuda", dtype=torch.float32)
    st = torch.zeros(B * Hv, device="cuda", dtype=torch.int32)
    gdn.gdn_decode_step_ab(d, w, G.dev(c.x), G.dev(c.z), G.dev(pc.hidden), G.dev(pc.W_a), G.dev(pc.W_b), conv, S,
                           out, dev_status=st)
    torch.cuda.synchronize()
    _, _, a64, b64 = oracle.in_proj(pc.hidden, pc.W_qkv, pc.W_z, pc.W_a, pc.W_b)
    ref = oracle.forward(Hk, Hv, c.x, c.z, a64, b64, c.conv_w, c.dt_bias, c.ssm_a, c.norm_w, c.conv0, S0.float(),
                         cu_seqlens=np.arange(B + 1))
    G.assert_out_close(out, ref.out, c.act_dtype)
    assert S.dtype == torch.bfloat16
    G.assert_state_one_rounding(S, ref.S)
    assert G.conv_bits_equal(conv, ref.conv_state, c.act_dtype)
    assert int(st.abs().sum()) == 0
