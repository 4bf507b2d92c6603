"""GPU parity on the method's degenerate cases, element by element against
the fp64 oracle through the C ABI (tolerances: tests/gpu_util.py).

The cases come from the layer definition on the xwen CLAUDE.md page
("Architecture cheat sheet", "Gated DeltaNet layer"):
  - beta = sigmoid(b_raw) at its ends: b_raw = +inf gives beta = 1 (the delta
    rule replaces the value stored under k), b_raw = -inf gives beta = 0 (the
    token writes nothing, the state only decays);
  - strong decay: ssm_a = -16 (the most negative value of the workloads'
    ssm_a = -exp(U(0, ln 16))) with a_raw = 3, so g is about -20 to -65 per
    token and the cumulative decay inside a 64-token chunk reaches about
    -4000 (the chunked form must not form e^{+Gam} or e^{-Gam} alone);
  - the clamp form of the L2 norm, x / max(||x||, eps): a q head whose conv
    taps are zero (q = 0, so q_hat = 0 and o = 0, not NaN) and a k head whose
    taps are scaled by 1e-8 (||k|| < eps, so k_hat = k / eps, not a unit
    vector).
Each runs through the chunked prefill (tensor-core and fp32 CUDA-core
kernels), the decode step (cluster and streaming kernels) and the verify walk.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_decode_gb300 as gdn
import gdn_inputs
import oracle
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def make_edge(c):
    """Apply the degenerate inputs to case c in place (c has H_k >= 2, H_v >= 2)."""
    D = 128
    T, Hk = c.T, c.Hk
    b = c.b_raw.float()
    b[0::2, 0] = float("inf")            # v-head 0: beta = 1 on even tokens,
    b[1::2, 0] = float("-inf")           #           beta = 0 on odd ones
    c.b_raw = b.to(c.act_dtype)
    a = c.a_raw.float()
    a[:, 1] = 3.0                        # v-head 1: strong decay
    c.a_raw = a.to(c.act_dtype)
    c.ssm_a = c.ssm_a.clone()
    c.ssm_a[1] = -16.0
    c.conv_w = c.conv_w.clone()
    c.conv_w[0:D] = 0.0                  # q of q/k head 0: zero vector
    c.conv_w[Hk * D + D:Hk * D + 2 * D] *= 1e-8   # k of q/k head 1: norm below eps
    return c


def oracle_prefill(c):
    return oracle.forward(c.Hk, c.Hv, c.x, c.z, c.a_raw, c.b_raw, c.conv_w, c.dt_bias, c.ssm_a, c.norm_w,
                          c.conv0, c.S0, cu_seqlens=c.cu_seqlens.numpy())


def check(c, out, pre, conv, S, ref):
    G.assert_out_close(out, ref.out, c.act_dtype)
    G.assert_state_close(S, ref.S, c.act_dtype)
    assert G.conv_bits_equal(conv, ref.conv_state, c.act_dtype)
    # the zero-q head (v-heads tiled onto q/k head 0) outputs exactly zero
    pre = pre.cpu().view(c.T, c.Hv, 128)
    assert torch.count_nonzero(pre[:, 0::c.Hk]) == 0
    assert np.all(ref.prenorm.reshape(c.T, c.Hv, 128)[:, 0::c.Hk] == 0.0)


@pytest.mark.parametrize("act,fp32_path", [(torch.bfloat16, False), (torch.bfloat16, True), (torch.float32, False)],
                         ids=["bf16_tensor_core", "bf16_cuda_core", "fp32"])
def test_prefill_edge_cases(act, fp32_path):
    c = make_edge(gdn_inputs.make_case("edge_prefill", Hk=2, Hv=6, lengths=[150, 77, 64], act_dtype=act,
                                       seed=4401))
    d, w = G.dims(c, prefill_fp32=fp32_path), G.weights(c)
    cu = c.cu_seqlens.to(torch.int32).contiguous()
    conv, S = G.dev(c.conv0), G.dev(c.S0)
    out = torch.empty(c.T, c.Hv * 128, device="cuda")
    pre = torch.empty(c.T, c.Hv * 128, device="cuda")
    nws = gdn.gdn_prefill_workspace_bytes(d, c.N, c.T)
    ws = torch.empty(max(nws, 16), device="cuda", dtype=torch.uint8) if nws else None
    gdn.gdn_prefill_chunked(d, w, cu, G.dev(cu), G.dev(c.x), G.dev(c.z), G.dev(c.a_raw), G.dev(c.b_raw), conv, S,
                            out, prenorm_out=pre, workspace=ws)
    torch.cuda.synchronize()
    check(c, out, pre, conv, S, oracle_prefill(c))


@pytest.mark.parametrize("B,Hk,Hv,act", [(3, 2, 6, torch.bfloat16), (3, 2, 4, torch.float32),
                                         (64, 16, 32, torch.bfloat16)],
                         ids=["cluster_bf16", "cluster_fp32", "stream_bf16"])
def test_decode_edge_cases(B, Hk, Hv, act):
    c = make_edge(gdn_inputs.make_case("edge_decode", Hk=Hk, Hv=Hv, B=B, K=1, act_dtype=act, seed=4402 + B))
    d, w = G.dims(c), G.weights(c)
    conv, S = G.dev(c.conv0), G.dev(c.S0)
    out = torch.empty(B, c.Hv * 128, device="cuda")
    pre = torch.empty(B, c.Hv * 128, device="cuda")
    gdn.gdn_decode_step(d, w, G.dev(c.x), G.dev(c.z), G.dev(c.a_raw), G.dev(c.b_raw), conv, S, out, pre)
    torch.cuda.synchronize()
    check(c, out, pre, conv, S, oracle_prefill(c))


@pytest.mark.parametrize("B,Hk,Hv", [(3, 2, 6), (64, 16, 32)], ids=["cluster", "stream"])
def test_verify_edge_cases(B, Hk, Hv):
    K = 3
    c = make_edge(gdn_inputs.make_case("edge_verify", Hk=Hk, Hv=Hv, B=B, K=K, seed=4403 + B))
    d, w = G.dims(c), G.weights(c)
    ck_conv = torch.empty(B, K, 3, c.C, device="cuda", dtype=c.act_dtype)
    ck_S = torch.empty(B, K, c.Hv, 128, 128, device="cuda")
    out = torch.empty(B * K, c.Hv * 128, device="cuda")
    gdn.gdn_verify_k(d, w, K, G.dev(c.x), G.dev(c.z), G.dev(c.a_raw), G.dev(c.b_raw), G.dev(c.conv0),
                     G.dev(c.S0), ck_conv, ck_S, out)
    torch.cuda.synchronize()
    o_ref, _, S_ck, c_ck = oracle.verify_checkpoints(c.Hk, c.Hv, c.x, c.z, c.a_raw, c.b_raw, c.conv_w, c.dt_bias,
                                                     c.ssm_a, c.norm_w, c.conv0, c.S0, K)
    G.assert_out_close(out, o_ref, c.act_dtype)
    assert G.conv_bits_equal(ck_conv, c_ck, c.act_dtype)
    for p in range(K):
        G.assert_state_close(ck_S[:, p], S_ck[:, p], c.act_dtype)
