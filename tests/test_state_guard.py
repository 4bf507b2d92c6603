"""GPU tests of the non-finite state guard: the status summary with its
listing cap (gdn_state_faults) and the reset of faulted states
(gdn_state_reset), on plain states and on a state ring.  A fault is planted
as a NaN in one v-head's channels of the input, on the host."""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_decode_gb300 as gdn
import gdn_inputs
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

FAULTS = [(7, 3), (20, 10), (41, 31)]      # (sequence, v-head) of the planted faults


def _plant(c, faults):
    """NaN in channel 5 of v-head h of sequence n (v channels follow the 2*H_k*128 q/k channels)."""
    for n, h in faults:
        c.x[n, 2 * c.Hk * 128 + h * 128 + 5] = float("nan")


@pytest.mark.parametrize("cap", [0, 2, 3, 1000])
def test_faults_summary_of_random_words(cap):
    """Summary against numpy over 4,800 words (five tiles of the walk), sparse nonzero bits."""
    g = torch.Generator().manual_seed(3 + cap)
    N, Hv = 100, 48
    st = torch.zeros(N * Hv, dtype=torch.int32)
    idx = torch.randperm(N * Hv, generator=g)[:37]
    st[idx] = torch.randint(1, 20, (37,), generator=g, dtype=torch.int32)
    d = gdn.make_dims(16, Hv, torch.bfloat16, torch.bfloat16, check_finite=True)
    rep = gdn.gdn_state_faults(d, st.cuda(), cap).cpu().numpy()
    nz = np.flatnonzero(st.numpy())
    assert rep[0] == len(nz) and rep[1] == min(len(nz), cap)
    k = rep[1]
    assert np.array_equal(rep[2:2 + 2 * k:2], nz[:k])
    assert np.array_equal(rep[3:3 + 2 * k:2], st.numpy()[nz[:k]])


def test_guard_detects_summarises_and_resets():
    c = gdn_inputs.make_case("guard", Hk=16, Hv=32, B=64, K=1, seed=77)
    _plant(c, FAULTS)
    d = G.dims(c, torch.bfloat16, check_finite=True)
    w = G.weights(c)
    conv, S = G.dev(c.conv0), G.dev(c.S0)
    out = torch.empty(64, c.Hv * 128, device="cuda", dtype=torch.bfloat16)
    st = torch.zeros(64 * c.Hv, dtype=torch.int32, device="cuda")
    gdn.gdn_decode_step(d, w, G.dev(c.x), G.dev(c.z), G.dev(c.a_raw), G.dev(c.b_raw), conv, S, out, None, st)
    torch.cuda.synchronize()
    want = sorted(n * c.Hv + h for n, h in FAULTS)
    rep = gdn.gdn_state_faults(d, st, 2).cpu().tolist()
    assert rep[0] == 3 and rep[1] == 2
    assert rep[2:] == [want[0], 3, want[1], 3]          # bit 0 state, bit 1 output
    rep = gdn.gdn_state_faults(d, st, 8).cpu().tolist()
    assert rep[:2] == [3, 3] and rep[2:8:2] == want
    S_before, conv_before = S.clone(), conv.clone()
    gdn.gdn_state_reset(d, S, st, conv_state=conv)
    torch.cuda.synchronize()
    assert int(st.abs().sum()) == 0
    bad_seq = {n for n, _ in FAULTS}
    for n in range(64):
        for h in range(c.Hv):
            if (n, h) in FAULTS:
                assert int(torch.count_nonzero(S[n, h])) == 0
            else:
                assert torch.equal(S[n, h], S_before[n, h])
        if n in bad_seq:
            assert int(torch.count_nonzero(conv[n])) == 0
        else:
            assert torch.equal(conv[n], conv_before[n])
    # the next step with finite inputs runs clean
    x2 = G.dev(gdn_inputs.make_case("guard2", Hk=16, Hv=32, B=64, K=1, seed=78).x)
    gdn.gdn_decode_step(d, w, x2, G.dev(c.z), G.dev(c.a_raw), G.dev(c.b_raw), conv, S, out, None, st)
    torch.cuda.synchronize()
    assert int(st.abs().sum()) == 0 and bool(torch.isfinite(S).all()) and bool(torch.isfinite(out.float()).all())


def test_reset_on_a_ring_zeroes_the_live_slot_only():
    B, R = 3, 4
    c = gdn_inputs.make_case("guard_ring", Hk=2, Hv=4, B=B, K=1, seed=79)
    _plant(c, [(1, 2)])
    d = G.dims(c, torch.float32, check_finite=True)
    w = G.weights(c)
    cur = torch.tensor([0, 2, 3], dtype=torch.int32, device="cuda")
    S_ring = torch.randn(B, R, c.Hv, 128, 128, device="cuda")
    S_ring[torch.arange(B, device="cuda"), cur.long()] = G.dev(c.S0)
    conv = G.dev(c.conv0)
    out = torch.empty(B, c.Hv * 128, device="cuda")
    st = torch.zeros(B * c.Hv, dtype=torch.int32, device="cuda")
    gdn.gdn_decode_step_ring(d, w, G.dev(c.x), G.dev(c.z), G.dev(c.a_raw), G.dev(c.b_raw), conv, S_ring, cur,
                             out, None, st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0] * 6 + [3] + [0] * 5
    before = S_ring.clone()
    gdn.gdn_state_reset(d, S_ring, st, ring_cur=cur)
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(S_ring[1, 2, 2])) == 0
    S_ring[1, 2, 2] = before[1, 2, 2]
    assert torch.equal(S_ring.isnan(), before.isnan())
    assert torch.equal(torch.nan_to_num(S_ring), torch.nan_to_num(before))
    assert int(st.abs().sum()) == 0
