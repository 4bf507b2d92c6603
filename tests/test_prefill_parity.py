"""GPU parity of the chunked (chunk = 64) prefill against the fp64 oracle,
through the C ABI: the tiny fp32 case (both forms), the T=8192 prefill
workload at full size, the packed varlen workload on sampled sequences,
ragged/empty sequences, split-and-resume, and zero_init.
Tolerances: tests/gpu_util.py."""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_decode_gb300 as gdn
import gdn_inputs
import oracle
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def run_prefill(c, zero_init=False, out_dtype=torch.float32, conv=None, S=None, check_finite=False,
                prefill_fp32=False):
    d, w = G.dims(c, out_dtype, check_finite, prefill_fp32), G.weights(c)
    cu = c.cu_seqlens.to(torch.int32).contiguous()
    conv = G.dev(c.conv0 if conv is None else conv)
    S = G.dev(c.S0 if S is None else S)
    out = torch.empty(c.T, c.Hv * 128, device="cuda", dtype=out_dtype)
    pre = torch.empty(c.T, c.Hv * 128, device="cuda")
    ws_bytes = gdn.gdn_prefill_workspace_bytes(d, c.N, c.T)
    ws = torch.empty(max(ws_bytes, 16), device="cuda", dtype=torch.uint8) if ws_bytes else None
    st = torch.zeros(c.N * c.Hv, device="cuda", dtype=torch.int32) if check_finite else None
    gdn.gdn_prefill_chunked(d, w, cu, G.dev(cu), G.dev(c.x), G.dev(c.z), G.dev(c.a_raw), G.dev(c.b_raw), conv, S,
                            out, zero_init=zero_init, prenorm_out=pre, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    return out, pre, conv, S, st


def oracle_run(c, conv0=None, S0=None, seqs=None):
    conv0 = c.conv0 if conv0 is None else conv0
    S0 = c.S0 if S0 is None else S0
    return oracle.forward(c.Hk, c.Hv, c.x, c.z, c.a_raw, c.b_raw, c.conv_w, c.dt_bias, c.ssm_a, c.norm_w,
                          conv0, S0, cu_seqlens=c.cu_seqlens.numpy())


def test_tiny_fp32_both_forms():
    """Tiny case (T=128, H_k=2, H_v=4, fp32): chunked prefill and T decode
    steps both match the oracle to 1e-5."""
    c = gdn_inputs.tiny_fp32()
    out, pre, conv, S, _ = run_prefill(c, zero_init=True)
    ref = oracle_run(c)
    G.assert_out_close(out, ref.out, torch.float32)
    G.assert_state_close(S, ref.S, torch.float32)
    assert G.conv_bits_equal(conv, ref.conv_state, torch.float32)
    # recurrent form: T decode steps of a batch of one
    d, w = G.dims(c), G.weights(c)
    conv_d, S_d = G.dev(c.conv0), G.dev(c.S0)
    outs = []
    for t in range(c.T):
        o = torch.empty(1, c.Hv * 128, device="cuda")
        gdn.gdn_decode_step(d, w, G.dev(c.x[t:t + 1]), G.dev(c.z[t:t + 1]), G.dev(c.a_raw[t:t + 1]),
                            G.dev(c.b_raw[t:t + 1]), conv_d, S_d, o)
        outs.append(o)
    torch.cuda.synchronize()
    G.assert_out_close(torch.cat(outs), ref.out, torch.float32)
    G.assert_state_close(S_d, ref.S, torch.float32)
    assert G.conv_bits_equal(conv_d, ref.conv_state, torch.float32)


@pytest.mark.parametrize("fp32_path", [False, True], ids=["tensor_core", "cuda_core"])
def test_prefill_t8192_full_size(fp32_path):
    """The prefill workload at full size (T=8192, 16/48, bf16, zero state),
    through the tensor-core kernel and the fp32 CUDA-core kernel."""
    c = gdn_inputs.prefill_t8192()
    out, pre, conv, S, _ = run_prefill(c, zero_init=True, prefill_fp32=fp32_path)
    ref = oracle_run(c)
    G.assert_out_close(out, ref.out, c.act_dtype)
    G.assert_state_close(S, ref.S, c.act_dtype)
    assert G.conv_bits_equal(conv, ref.conv_state, c.act_dtype)


@pytest.mark.parametrize("lengths", [[1, 63, 64, 65, 130, 0, 2], [200], [3, 3, 3]])
@pytest.mark.parametrize("act", [torch.bfloat16, torch.float32])
def test_ragged_varlen_nonzero_state(lengths, act):
    c = gdn_inputs.make_case("rag", Hk=2, Hv=6, lengths=lengths, act_dtype=act, seed=len(lengths) * 7 + sum(lengths))
    out, pre, conv, S, _ = run_prefill(c)
    ref = oracle_run(c)
    G.assert_out_close(out, ref.out, act)
    G.assert_state_close(S, ref.S, act)
    assert G.conv_bits_equal(conv, ref.conv_state, act)


def test_zero_init_ignores_state_buffers():
    c = gdn_inputs.make_case("zi", Hk=2, Hv=4, lengths=[70, 5], seed=3)
    garbage_S = torch.full_like(c.S0, float("nan"))
    garbage_c = torch.full_like(c.conv0, float("nan"))
    out, _, conv, S, _ = run_prefill(c, zero_init=True, conv=garbage_c, S=garbage_S)
    ref = oracle_run(c, conv0=torch.zeros_like(c.conv0), S0=torch.zeros_like(c.S0))
    G.assert_out_close(out, ref.out, c.act_dtype)
    G.assert_state_close(S, ref.S, c.act_dtype)
    assert G.conv_bits_equal(conv, ref.conv_state, c.act_dtype)


def test_split_and_resume():
    """Prefill of T1 tokens, then T2 more from the returned states, equals the
    oracle over T1 + T2 (the state carries across calls)."""
    c = gdn_inputs.make_case("sr", Hk=2, Hv=4, lengths=[150], seed=4)
    T1 = 77
    first = gdn_inputs.Case(**{**c.__dict__, "x": c.x[:T1], "z": c.z[:T1], "a_raw": c.a_raw[:T1],
                               "b_raw": c.b_raw[:T1], "cu_seqlens": torch.tensor([0, T1], dtype=torch.int32)})
    o1, _, conv, S, _ = run_prefill(first)
    second = gdn_inputs.Case(**{**c.__dict__, "x": c.x[T1:], "z": c.z[T1:], "a_raw": c.a_raw[T1:],
                                "b_raw": c.b_raw[T1:], "cu_seqlens": torch.tensor([0, 150 - T1], dtype=torch.int32)})
    o2, _, conv, S, _ = run_prefill(second, conv=conv.cpu(), S=S.cpu())
    ref = oracle_run(c)
    G.assert_out_close(torch.cat([o1, o2]), ref.out, c.act_dtype)
    G.assert_state_close(S, ref.S, c.act_dtype)
    assert G.conv_bits_equal(conv, ref.conv_state, c.act_dtype)


def test_prefill_in_segments_is_bit_identical():
    """A sequence prefilled in four calls of 256 tokens (zero initial state in the first, the
    conv and recurrent state carried on the device through the others) gives the outputs, the
    final state and the conv state of one call over all 1024 tokens bit for bit: the chunk
    grid is the same (256 is a multiple of 64), so is every operation.  (The bench's end-to-end
    leg streams its prefill this way to overlap the host copies.)"""
    c = gdn_inputs.make_case("seg", Hk=4, Hv=12, lengths=[1024], S0="zero", conv0="zero", seed=31)
    d, w = G.dims(c, torch.bfloat16), G.weights(c)
    dev = lambda t: G.dev(t)
    x, z, a, b = dev(c.x), dev(c.z), dev(c.a_raw), dev(c.b_raw)

    def run(segs):
        conv = torch.zeros(1, 3, c.C, device="cuda", dtype=torch.bfloat16)
        S = torch.zeros(1, c.Hv, 128, 128, device="cuda")
        out = torch.empty(c.T, c.Hv * 128, device="cuda", dtype=torch.bfloat16)
        L = c.T // segs
        cu_h = torch.tensor([0, L], dtype=torch.int32)
        ws = torch.empty(gdn.gdn_prefill_workspace_bytes(d, 1, L), device="cuda", dtype=torch.uint8)
        for i in range(segs):
            sl = slice(i * L, (i + 1) * L)
            gdn.gdn_prefill_chunked(d, w, cu_h, G.dev(cu_h), x[sl], z[sl], a[sl], b[sl], conv, S, out[sl],
                                    zero_init=(i == 0), workspace=ws)
        torch.cuda.synchronize()
        return out, S, conv

    one, four = run(1), run(4)
    for u, v in zip(one, four):
        assert torch.equal(u, v)


def test_varlen_t65536_all_sequences():
    """The packed varlen workload (8 sequences, T=65536, nonzero initial
    state) at full size on the GPU, in the launch configuration the bench
    times; the oracle recomputes all 8 sequences (every output, final state
    and conv state is compared)."""
    c = gdn_inputs.varlen_t65536()
    out, _, conv, S, _ = run_prefill(c)
    ref = oracle.forward(c.Hk, c.Hv, c.x, c.z, c.a_raw, c.b_raw, c.conv_w, c.dt_bias, c.ssm_a, c.norm_w,
                         c.conv0, c.S0, cu_seqlens=c.cu_seqlens.numpy())
    G.assert_out_close(out, ref.out, c.act_dtype)
    G.assert_state_close(S, ref.S, c.act_dtype)
    assert G.conv_bits_equal(conv, ref.conv_state, c.act_dtype)


@pytest.mark.parametrize("Hk,Hv,lengths", [(1, 1, [64]), (1, 3, [1]), (4, 8, [127, 65]), (2, 32, [300]),
                                            (3, 3, [5, 200, 64, 63]), (8, 96, [200, 70])])
def test_tensor_core_prefill_shapes(Hk, Hv, lengths):
    """Tensor-core prefill across head ratios 1..16, one-token and
    whole-chunk sequences, against the oracle.  96 v-heads over two sequences
    is more chains than the kernel gives chain CTAs (each CTA then walks
    several (sequence, v-head) chains, without the records-in-flight gate)."""
    c = gdn_inputs.make_case("tcs", Hk=Hk, Hv=Hv, lengths=lengths, seed=Hk * 31 + Hv + sum(lengths))
    out, pre, conv, S, _ = run_prefill(c)
    ref = oracle_run(c)
    G.assert_out_close(out, ref.out, c.act_dtype)
    G.assert_state_close(S, ref.S, c.act_dtype)
    assert G.conv_bits_equal(conv, ref.conv_state, c.act_dtype)


def test_prefill_bf16_output():
    c = gdn_inputs.make_case("bo", Hk=2, Hv=4, lengths=[100, 29], seed=8)
    out, _, _, _, _ = run_prefill(c, out_dtype=torch.bfloat16)
    ref = oracle_run(c)
    G.assert_out_close_bf16out(out, ref.out, c.act_dtype)


def test_prefill_nonfinite_reported():
    c = gdn_inputs.make_case("nf", Hk=2, Hv=4, lengths=[10, 10], seed=12)
    c.x[13, 2 * 256 + 128 + 3] = float("inf")     # sequence 1, v channel of head 1
    _, _, _, _, st = run_prefill(c, check_finite=True)
    st = st.cpu().view(2, 4)
    assert st[1, 1] != 0 and int((st != 0).sum()) == 1
