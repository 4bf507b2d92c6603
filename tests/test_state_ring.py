"""GPU tests of the state ring (gdn_verify_k_ring / gdn_commit_ring /
gdn_decode_step_ring): over several speculative rounds the ring path gives
bit for bit the outputs, checkpoints and live state of the copying
verify + commit path, reads only the live slot and writes only the slots
after it; and over several rounds it matches the fp64 oracle's verify walk
and commits directly."""
import pytest
import torch

import gated_deltanet_linear_decode_gb300 as gdn
import gdn_inputs
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def _round_slice(t, B, rounds, K, r):
    """Tokens r*K .. r*K+K-1 of every sequence from a [B*rounds*K, ...] draw, as [B*K, ...]."""
    v = t.view(B, rounds * K, *t.shape[1:])[:, r * K:(r + 1) * K]
    return G.dev(v.reshape(B * K, *t.shape[1:]).contiguous())


@pytest.mark.parametrize("B,Hk,Hv,K,R,act", [
    (64, 16, 32, 3, 4, torch.bfloat16),     # the streaming kernel; R = K + 1
    (64, 16, 32, 2, 5, torch.float32),      # R > K + 1: slots wrap at different points
    (3, 2, 4, 4, 5, torch.bfloat16),        # the cluster kernel
    (5, 2, 8, 1, 2, torch.float32),
])
def test_ring_rounds_equal_copy_path(B, Hk, Hv, K, R, act):
    rounds = 4
    c = gdn_inputs.make_case("ring", Hk=Hk, Hv=Hv, B=B, K=rounds * K, act_dtype=act, seed=70 + B + K)
    d, w = G.dims(c), G.weights(c)
    gen = torch.Generator().manual_seed(5)
    # copying path
    conv, S = G.dev(c.conv0), G.dev(c.S0)
    ck_conv = torch.empty(B, K, 3, c.C, device="cuda", dtype=act)
    ck_S = torch.empty(B, K, c.Hv, 128, 128, device="cuda")
    out = torch.empty(B * K, c.Hv * 128, device="cuda")
    # ring path: slot 0 live, the other slots poisoned so a stray read shows
    conv_r = G.dev(c.conv0)
    S_ring = torch.full((B, R, c.Hv, 128, 128), float("nan"), device="cuda")
    S_ring[:, 0] = G.dev(c.S0)
    cur = torch.zeros(B, dtype=torch.int32, device="cuda")
    ck_conv_r = torch.empty_like(ck_conv)
    out_r = torch.empty_like(out)
    for r in range(rounds):
        x, z = _round_slice(c.x, B, rounds, K, r), _round_slice(c.z, B, rounds, K, r)
        a, b = _round_slice(c.a_raw, B, rounds, K, r), _round_slice(c.b_raw, B, rounds, K, r)
        acc = torch.randint(1, K + 1, (B,), generator=gen, dtype=torch.int32)
        if r == 2:
            acc[0] = 0                      # out of range: the sequence keeps its state
            acc[-1] = K + 1
        acc = acc.cuda()
        gdn.gdn_verify_k(d, w, K, x, z, a, b, conv, S, ck_conv, ck_S, out)
        gdn.gdn_commit(d, K, acc, ck_conv, ck_S, conv, S)
        cur0 = cur.clone()
        gdn.gdn_verify_k_ring(d, w, K, x, z, a, b, conv_r, S_ring, cur, ck_conv_r, out_r)
        torch.cuda.synchronize()
        assert torch.equal(out_r, out) and torch.equal(ck_conv_r, ck_conv)
        for bb in range(B):
            for p in range(K):
                assert torch.equal(S_ring[bb, (int(cur0[bb]) + 1 + p) % R], ck_S[bb, p])
        gdn.gdn_commit_ring(d, K, R, acc, ck_conv_r, conv_r, cur)
        torch.cuda.synchronize()
        n = acc.cpu()
        exp_cur = torch.where((n >= 1) & (n <= K), (cur0.cpu() + n) % R, cur0.cpu())
        assert torch.equal(cur.cpu(), exp_cur)
        assert torch.equal(conv_r, conv)
        for bb in range(B):
            assert torch.equal(S_ring[bb, int(exp_cur[bb])], S[bb])


@pytest.mark.parametrize("B,Hk,Hv,act", [(64, 16, 32, torch.bfloat16), (2, 2, 4, torch.float32)])
def test_decode_step_ring_equals_decode_step(B, Hk, Hv, act):
    steps, R = 3, 3
    c = gdn_inputs.make_case("rdec", Hk=Hk, Hv=Hv, B=B, K=steps, act_dtype=act, seed=90 + B)
    d, w = G.dims(c), G.weights(c)
    conv, S = G.dev(c.conv0), G.dev(c.S0)
    conv_r = G.dev(c.conv0)
    cur = (torch.arange(B, dtype=torch.int32) % R).cuda()
    S_ring = torch.full((B, R, c.Hv, 128, 128), float("nan"), device="cuda")
    S_ring[torch.arange(B, device="cuda"), cur.long()] = S
    ring0 = S_ring.clone()
    for t in range(steps):
        x, z = _round_slice(c.x, B, 1, steps, 0).view(B, steps, -1)[:, t].contiguous(), \
            _round_slice(c.z, B, 1, steps, 0).view(B, steps, -1)[:, t].contiguous()
        a = G.dev(c.a_raw.view(B, steps, -1)[:, t].contiguous())
        b = G.dev(c.b_raw.view(B, steps, -1)[:, t].contiguous())
        o = torch.empty(B, c.Hv * 128, device="cuda")
        o_r = torch.empty_like(o)
        gdn.gdn_decode_step(d, w, x, z, a, b, conv, S, o)
        gdn.gdn_decode_step_ring(d, w, x, z, a, b, conv_r, S_ring, cur, o_r)
        torch.cuda.synchronize()
        assert torch.equal(o_r, o) and torch.equal(conv_r, conv)
        for bb in range(B):
            k = int(cur[bb])
            assert torch.equal(S_ring[bb, k], S[bb])
            for j in range(R):
                if j != k:                  # the other slots are not touched
                    assert torch.equal(S_ring[bb, j].isnan(), ring0[bb, j].isnan())
    assert torch.equal(cur.cpu(), torch.arange(B, dtype=torch.int32) % R)


@pytest.mark.parametrize("B,Hk,Hv,K,R,act", [
    (64, 16, 32, 3, 4, torch.bfloat16),     # the streaming kernel (the verify workload's shape)
    (3, 2, 4, 4, 6, torch.float32),         # the cluster kernel, R > K + 1
])
def test_ring_rounds_match_oracle(B, Hk, Hv, K, R, act):
    """Three speculative rounds on the state ring against the fp64 oracle's
    verify walk (checkpoint p = the state after draft position p; accept n
    makes checkpoint n - 1 the live state), the oracle carrying its own
    committed states from round to round: outputs, every checkpoint slot, the
    live slot after each commit (tolerances of tests/gpu_util.py) and the conv
    checkpoints and conv state (bit for bit)."""
    import numpy as np
    import oracle
    rounds = 3
    c = gdn_inputs.make_case("ring_oracle", Hk=Hk, Hv=Hv, B=B, K=rounds * K, act_dtype=act, seed=310 + B)
    d, w = G.dims(c), G.weights(c)
    gen = torch.Generator().manual_seed(11)
    conv_r = G.dev(c.conv0)
    S_ring = torch.full((B, R, c.Hv, 128, 128), float("nan"), device="cuda")
    S_ring[:, 0] = G.dev(c.S0)
    cur = torch.zeros(B, dtype=torch.int32, device="cuda")
    ck_conv = torch.empty(B, K, 3, c.C, device="cuda", dtype=act)
    out = torch.empty(B * K, c.Hv * 128, device="cuda")
    conv_ref, S_ref = c.conv0.float().numpy(), c.S0.double().numpy()
    rows = lambda t, r: t.view(B, rounds * K, *t.shape[1:])[:, r * K:(r + 1) * K].reshape(B * K, *t.shape[1:])
    for r in range(rounds):
        x, z, a, b = (rows(t, r).contiguous() for t in (c.x, c.z, c.a_raw, c.b_raw))
        acc = torch.randint(1, K + 1, (B,), generator=gen, dtype=torch.int32)
        cur0 = cur.cpu().numpy().copy()
        gdn.gdn_verify_k_ring(d, w, K, G.dev(x), G.dev(z), G.dev(a), G.dev(b), conv_r, S_ring, cur, ck_conv, out)
        gdn.gdn_commit_ring(d, K, R, acc.cuda(), ck_conv, conv_r, cur)
        torch.cuda.synchronize()
        o_ref, _, S_ck, c_ck = oracle.verify_checkpoints(Hk, Hv, x, z, a, b, c.conv_w, c.dt_bias, c.ssm_a,
                                                         c.norm_w, conv_ref, S_ref, K)
        G.assert_out_close(out, o_ref, act)
        assert G.conv_bits_equal(ck_conv, c_ck, act)
        ring = S_ring.cpu()
        for p in range(K):
            slots = torch.from_numpy((cur0 + 1 + p) % R)
            G.assert_state_close(ring[torch.arange(B), slots], S_ck[:, p], act)
        n = acc.numpy()
        S_ref = S_ck[np.arange(B), n - 1]
        conv_ref = c_ck[np.arange(B), n - 1]
        assert np.array_equal(cur.cpu().numpy(), (cur0 + n) % R)
        G.assert_state_close(ring[torch.arange(B), cur.cpu().long()], S_ref, act)
        assert G.conv_bits_equal(conv_r, conv_ref, act)
