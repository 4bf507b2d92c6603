"""GPU parity of the recurrent path (decode step, verify walk, commit) against
the fp64 oracle, through the C ABI.  Tolerances: tests/gpu_util.py."""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_decode_gb300 as gdn
import gdn_inputs
import oracle
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def _oracle_decode(c, x, z, a, b, conv, S):
    B = conv.shape[0]
    return oracle.forward(c.Hk, c.Hv, x, z, a, b, c.conv_w, c.dt_bias, c.ssm_a, c.norm_w, conv, S,
                          cu_seqlens=np.arange(B + 1))


def _decode(c, out_dtype=torch.float32, check_finite=False, x=None, conv=None, S=None):
    d = G.dims(c, out_dtype, check_finite)
    w = G.weights(c)
    B = c.N
    x = G.dev(c.x if x is None else x)
    conv = G.dev(c.conv0 if conv is None else conv)
    S = G.dev(c.S0 if S is None else S)
    out = torch.empty(B, c.Hv * 128, device="cuda", dtype=out_dtype)
    pre = torch.empty(B, c.Hv * 128, device="cuda", dtype=torch.float32)
    st = torch.zeros(B * c.Hv, device="cuda", dtype=torch.int32)
    gdn.gdn_decode_step(d, w, x, G.dev(c.z), G.dev(c.a_raw), G.dev(c.b_raw), conv, S, out, pre,
                        st if check_finite else None)
    torch.cuda.synchronize()
    return out, pre, conv, S, st


@pytest.mark.parametrize("maker", [gdn_inputs.decode_b64, gdn_inputs.decode_b1])
def test_decode_step_matches_oracle(maker):
    c = maker()
    out, pre, conv, S, _ = _decode(c)
    ref = _oracle_decode(c, c.x, c.z, c.a_raw, c.b_raw, c.conv0, c.S0)
    G.assert_out_close(out, ref.out, c.act_dtype)
    G.assert_state_close(S, ref.S, c.act_dtype)
    assert G.conv_bits_equal(conv, ref.conv_state, c.act_dtype)
    np.testing.assert_allclose(pre.cpu().numpy(), ref.prenorm, atol=1e-4, rtol=1e-3)


@pytest.mark.parametrize("Hk,Hv,act", [(2, 2, torch.bfloat16), (4, 12, torch.bfloat16), (2, 8, torch.bfloat16),
                                       (1, 16, torch.bfloat16), (2, 4, torch.float32), (16, 48, torch.bfloat16)])
def test_decode_head_ratios(Hk, Hv, act):
    """H_v/H_k = 1, 3, 4, 16 and 2 (cluster sizes 4, 6, 8, 16 and 8); fp32 path at 1e-5."""
    c = gdn_inputs.make_case("r", Hk=Hk, Hv=Hv, B=3, K=1, act_dtype=act, seed=Hk * 100 + Hv)
    out, pre, conv, S, _ = _decode(c)
    ref = _oracle_decode(c, c.x, c.z, c.a_raw, c.b_raw, c.conv0, c.S0)
    G.assert_out_close(out, ref.out, act)
    G.assert_state_close(S, ref.S, act)
    assert G.conv_bits_equal(conv, ref.conv_state, act)


def test_decode_many_steps_in_place():
    """24 in-place steps of a B=2 batch equal the oracle run over 24-token sequences."""
    steps, B = 24, 2
    c = gdn_inputs.make_case("seq", Hk=4, Hv=8, lengths=[steps] * B, seed=5)
    d, w = G.dims(c), G.weights(c)
    conv, S = G.dev(c.conv0), G.dev(c.S0)
    outs = []
    x = c.x.view(B, steps, -1); z = c.z.view(B, steps, -1)
    a = c.a_raw.view(B, steps, -1); b = c.b_raw.view(B, steps, -1)
    for t in range(steps):
        out = torch.empty(B, c.Hv * 128, device="cuda")
        gdn.gdn_decode_step(d, w, G.dev(x[:, t]), G.dev(z[:, t]), G.dev(a[:, t]), G.dev(b[:, t]), conv, S, out)
        outs.append(out)
    torch.cuda.synchronize()
    got = torch.stack(outs, 1).reshape(B * steps, -1)
    ref = oracle.forward(c.Hk, c.Hv, c.x, c.z, c.a_raw, c.b_raw, c.conv_w, c.dt_bias, c.ssm_a, c.norm_w,
                         c.conv0, c.S0, cu_seqlens=c.cu_seqlens)
    G.assert_out_close(got, ref.out, c.act_dtype)
    G.assert_state_close(S, ref.S, c.act_dtype)
    assert G.conv_bits_equal(conv, ref.conv_state, c.act_dtype)


def test_decode_bf16_output():
    c = gdn_inputs.decode_b64()
    out, _, _, _, _ = _decode(c, out_dtype=torch.bfloat16)
    ref = _oracle_decode(c, c.x, c.z, c.a_raw, c.b_raw, c.conv0, c.S0)
    G.assert_out_close_bf16out(out, ref.out, c.act_dtype)


def test_decode_recall_invariant_full_pipeline():
    """beta = 1 (b_raw = +inf) and the q channels equal to the k channels give
    o = v / sqrt(128) before the norm, for any state and decay."""
    c = gdn_inputs.make_case("inv", Hk=2, Hv=4, B=5, K=1, act_dtype=torch.float32, seed=9)
    c.b_raw[:] = float("inf")
    c.x[:, :256] = c.x[:, 256:512]
    c.conv_w[:256] = c.conv_w[256:512]
    c.conv0[:, :, :256] = c.conv0[:, :, 256:512]
    _, pre, _, _, _ = _decode(c)
    ref = oracle.forward(c.Hk, c.Hv, c.x, c.z, c.a_raw, c.b_raw, c.conv_w, c.dt_bias, c.ssm_a, c.norm_w, c.conv0,
                         c.S0, cu_seqlens=np.arange(6), want_inter=True)
    v = ref.inter[..., 256:384].reshape(5, -1)
    np.testing.assert_allclose(pre.cpu().numpy(), v / np.sqrt(128), atol=2e-6, rtol=1e-5)


def test_decode_empty_batch_is_noop():
    c = gdn_inputs.make_case("e", Hk=2, Hv=4, B=1, K=1)
    d, w = G.dims(c), G.weights(c)
    e = torch.empty(0, device="cuda")
    gdn.library()
    st = gdn.library().gdn_decode_step(d, w.struct(), 0, None, None, None, None, None, None, None, None, None,
                                       None)
    assert st == 0


def test_nonfinite_state_is_reported():
    """A NaN input for sequence 1 flags (1, h) in dev_status and nothing else."""
    c = gdn_inputs.make_case("nan", Hk=2, Hv=4, B=3, K=1, seed=11)
    c.x[1, 2 * 256 + 5] = float("nan")          # one v channel of head 0 -> row 5 of (1, 0)
    _, _, _, _, st = _decode(c, check_finite=True)
    st = st.cpu().view(3, 4)
    assert st[1, 0] == 3 and int(st.sum()) == 3


@pytest.mark.parametrize("K", [1, 3, 16])
def test_verify_checkpoints_bitexact_vs_decode_steps(K):
    """Checkpoint p of the verify walk is bit-identical to the state after p+1
    decode steps; outputs are bit-identical too; both match the oracle."""
    B = 4
    c = gdn_inputs.make_case("v", Hk=4, Hv=8, B=B, K=K, seed=20 + K)
    d, w = G.dims(c), G.weights(c)
    C = c.C
    conv0, S0 = G.dev(c.conv0), G.dev(c.S0)
    ck_conv = torch.empty(B, K, 3, C, device="cuda", dtype=c.act_dtype)
    ck_S = torch.empty(B, K, c.Hv, 128, 128, device="cuda")
    out = torch.empty(B * K, c.Hv * 128, device="cuda")
    gdn.gdn_verify_k(d, w, K, G.dev(c.x), G.dev(c.z), G.dev(c.a_raw), G.dev(c.b_raw), conv0, S0, ck_conv, ck_S, out)
    conv, S = conv0.clone(), S0.clone()
    xs = c.x.view(B, K, -1); zs = c.z.view(B, K, -1); as_ = c.a_raw.view(B, K, -1); bs = c.b_raw.view(B, K, -1)
    out_v = out.view(B, K, -1)
    for p in range(K):
        o = torch.empty(B, c.Hv * 128, device="cuda")
        gdn.gdn_decode_step(d, w, G.dev(xs[:, p]), G.dev(zs[:, p]), G.dev(as_[:, p]), G.dev(bs[:, p]), conv, S, o)
        torch.cuda.synchronize()
        assert torch.equal(ck_S[:, p], S), f"state checkpoint {p} differs from decode replay"
        assert torch.equal(ck_conv[:, p], conv), f"conv checkpoint {p} differs"
        assert torch.equal(out_v[:, p], o)
    # inputs untouched by the verify walk
    assert torch.equal(conv0.cpu(), c.conv0) and torch.equal(S0.cpu(), c.S0)
    o_ref, _, S_ck_ref, c_ck_ref = oracle.verify_checkpoints(c.Hk, c.Hv, c.x, c.z, c.a_raw, c.b_raw, c.conv_w,
                                                             c.dt_bias, c.ssm_a, c.norm_w, c.conv0, c.S0, K)
    G.assert_out_close(out, o_ref, c.act_dtype)
    G.assert_state_close(ck_S, S_ck_ref, c.act_dtype)
    assert G.conv_bits_equal(ck_conv, c_ck_ref, c.act_dtype)


@pytest.mark.parametrize("K,act", [(2, torch.bfloat16), (1, torch.float32), (5, torch.bfloat16)])
def test_large_batch_verify_bitexact_vs_decode(K, act):
    """At B*H_k of several items per SM the library takes its streaming
    (persistent) kernel for both calls; checkpoints still equal decode
    replays bit for bit and match the oracle."""
    B = 64
    c = gdn_inputs.make_case("lv", Hk=16, Hv=32, B=B, K=K, act_dtype=act, seed=40 + K)
    d, w = G.dims(c), G.weights(c)
    conv0, S0 = G.dev(c.conv0), G.dev(c.S0)
    ck_conv = torch.empty(B, K, 3, c.C, device="cuda", dtype=act)
    ck_S = torch.empty(B, K, c.Hv, 128, 128, device="cuda")
    out = torch.empty(B * K, c.Hv * 128, device="cuda")
    gdn.gdn_verify_k(d, w, K, G.dev(c.x), G.dev(c.z), G.dev(c.a_raw), G.dev(c.b_raw), conv0, S0, ck_conv, ck_S, out)
    conv, S = conv0.clone(), S0.clone()
    xs = c.x.view(B, K, -1); zs = c.z.view(B, K, -1); as_ = c.a_raw.view(B, K, -1); bs = c.b_raw.view(B, K, -1)
    for p in range(K):
        o = torch.empty(B, c.Hv * 128, device="cuda")
        gdn.gdn_decode_step(d, w, G.dev(xs[:, p]), G.dev(zs[:, p]), G.dev(as_[:, p]), G.dev(bs[:, p]), conv, S, o)
        torch.cuda.synchronize()
        assert torch.equal(ck_S[:, p], S) and torch.equal(ck_conv[:, p], conv)
        assert torch.equal(out.view(B, K, -1)[:, p], o)
    o_ref, _, S_ck_ref, c_ck_ref = oracle.verify_checkpoints(c.Hk, c.Hv, c.x, c.z, c.a_raw, c.b_raw, c.conv_w,
                                                             c.dt_bias, c.ssm_a, c.norm_w, c.conv0, c.S0, K)
    G.assert_out_close(out, o_ref, act)
    G.assert_state_close(ck_S, S_ck_ref, act)
    assert G.conv_bits_equal(ck_conv, c_ck_ref, act)


@pytest.mark.parametrize("B,Hk,Hv,K", [(19, 16, 32, 1), (23, 16, 32, 1), (37, 16, 48, 1), (23, 16, 32, 3), (41, 8, 24, 2)])
def test_streaming_kernel_uneven_groups(B, Hk, Hv, K):
    """Batches just above the streaming kernel's threshold: each CTA gets two or three
    (sequence, q/k head) groups, so its two compute groups carry unequal loads and share
    the stages unevenly.  The decode step against the oracle; the verify walk's
    checkpoints against decode replays bit for bit and the oracle."""
    c = gdn_inputs.make_case("ug", Hk=Hk, Hv=Hv, B=B, K=K, seed=5100 + B * K + Hv)
    d, w = G.dims(c), G.weights(c)
    conv0, S0 = G.dev(c.conv0), G.dev(c.S0)
    if K == 1:
        out, _, conv, S, _ = _decode(c)
        ref = oracle.forward(c.Hk, c.Hv, c.x, c.z, c.a_raw, c.b_raw, c.conv_w, c.dt_bias, c.ssm_a, c.norm_w,
                             c.conv0, c.S0, cu_seqlens=np.arange(B + 1))
        G.assert_out_close(out, ref.out, c.act_dtype)
        G.assert_state_close(S, ref.S, c.act_dtype)
        assert G.conv_bits_equal(conv, ref.conv_state, c.act_dtype)
        return
    ck_conv = torch.empty(B, K, 3, c.C, device="cuda", dtype=c.act_dtype)
    ck_S = torch.empty(B, K, c.Hv, 128, 128, device="cuda")
    out = torch.empty(B * K, c.Hv * 128, device="cuda")
    gdn.gdn_verify_k(d, w, K, G.dev(c.x), G.dev(c.z), G.dev(c.a_raw), G.dev(c.b_raw), conv0, S0, ck_conv, ck_S, out)
    conv, S = conv0.clone(), S0.clone()
    xs = c.x.view(B, K, -1); zs = c.z.view(B, K, -1); as_ = c.a_raw.view(B, K, -1); bs = c.b_raw.view(B, K, -1)
    for p in range(K):
        o = torch.empty(B, c.Hv * 128, device="cuda")
        gdn.gdn_decode_step(d, w, G.dev(xs[:, p]), G.dev(zs[:, p]), G.dev(as_[:, p]), G.dev(bs[:, p]), conv, S, o)
        torch.cuda.synchronize()
        assert torch.equal(ck_S[:, p], S) and torch.equal(ck_conv[:, p], conv)
        assert torch.equal(out.view(B, K, -1)[:, p], o)
    o_ref, _, S_ck_ref, c_ck_ref = oracle.verify_checkpoints(c.Hk, c.Hv, c.x, c.z, c.a_raw, c.b_raw, c.conv_w,
                                                             c.dt_bias, c.ssm_a, c.norm_w, c.conv0, c.S0, K)
    G.assert_out_close(out, o_ref, c.act_dtype)
    G.assert_state_close(ck_S, S_ck_ref, c.act_dtype)
    assert G.conv_bits_equal(ck_conv, c_ck_ref, c.act_dtype)


def test_large_batch_nonfinite_reported():
    c = gdn_inputs.make_case("lnan", Hk=16, Hv=32, B=64, K=1, seed=13)
    c.x[7, 2 * 16 * 128 + 3 * 128 + 9] = float("nan")     # sequence 7, v-head 3, row 9
    _, _, _, _, st = _decode(c, check_finite=True)
    st = st.cpu().view(64, 32)
    assert st[7, 3] == 3 and int((st != 0).sum()) == 1


def test_verify_b64_k3_commit():
    """The verify workload (B=64, K=3, 16/32, bf16): outputs and checkpoints vs
    the oracle; commit(accept_len) makes the live state bit-identical to
    accept_len decode steps."""
    c = gdn_inputs.verify_b64_k3()
    B, K = c.N, c.K
    d, w = G.dims(c), G.weights(c)
    conv0, S0 = G.dev(c.conv0), G.dev(c.S0)
    ck_conv = torch.empty(B, K, 3, c.C, device="cuda", dtype=c.act_dtype)
    ck_S = torch.empty(B, K, c.Hv, 128, 128, device="cuda")
    out = torch.empty(B * K, c.Hv * 128, device="cuda")
    gdn.gdn_verify_k(d, w, K, G.dev(c.x), G.dev(c.z), G.dev(c.a_raw), G.dev(c.b_raw), conv0, S0, ck_conv, ck_S, out)
    o_ref, _, S_ck_ref, c_ck_ref = oracle.verify_checkpoints(c.Hk, c.Hv, c.x, c.z, c.a_raw, c.b_raw, c.conv_w,
                                                             c.dt_bias, c.ssm_a, c.norm_w, c.conv0, c.S0, K)
    torch.cuda.synchronize()
    G.assert_out_close(out, o_ref, c.act_dtype)
    G.assert_state_close(ck_S, S_ck_ref, c.act_dtype)
    assert G.conv_bits_equal(ck_conv, c_ck_ref, c.act_dtype)
    acc = G.dev(c.accept_len)
    conv, S = conv0.clone(), S0.clone()
    gdn.gdn_commit(d, K, acc, ck_conv, ck_S, conv, S)
    torch.cuda.synchronize()
    for bb in range(B):
        n = int(c.accept_len[bb])
        assert torch.equal(S[bb], ck_S[bb, n - 1]) and torch.equal(conv[bb], ck_conv[bb, n - 1])
    # out-of-range accept lengths leave the state alone
    bad = torch.tensor([0, K + 1] + [1] * (B - 2), dtype=torch.int32, device="cuda")
    conv2, S2 = conv0.clone(), S0.clone()
    gdn.gdn_commit(d, K, bad, ck_conv, ck_S, conv2, S2)
    torch.cuda.synchronize()
    assert torch.equal(S2[:2], S0[:2]) and torch.equal(S2[2:], ck_S[2:, 0])


def test_conv_state_init():
    c = gdn_inputs.make_case("ci", Hk=2, Hv=4, B=3, K=1)
    d = G.dims(c)
    cs = torch.full((3, 3, c.C), 7.0, device="cuda", dtype=c.act_dtype)
    gdn.gdn_conv_state_init(d, cs)
    torch.cuda.synchronize()
    assert torch.count_nonzero(cs) == 0
    pre = G.dev(c.conv0)
    gdn.gdn_conv_state_init(d, cs, pre)
    torch.cuda.synchronize()
    assert torch.equal(cs, pre)
