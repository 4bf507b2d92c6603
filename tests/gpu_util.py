"""Helpers shared by the GPU parity tests: move a seeded case to the device,
compare against the oracle with the stated tolerances.

Tolerances (the layer's accuracy contract): bf16 activations -- max |y - y_ref|
<= 2e-3 over all outputs and ||S - S_ref||_F / ||S_ref||_F <= 1e-3 per
(sequence, head); fp32 activations -- both <= 1e-5.  Outputs are compared in
fp32; a bf16 output adds half a bf16 ulp of the reference value.  Conv-state
bookkeeping is compared bit for bit."""
import numpy as np
import torch

import gated_deltanet_linear_decode_gb300 as gdn

TOL = {torch.bfloat16: (2e-3, 1e-3), torch.float32: (1e-5, 1e-5)}


def dev(t):
    return t.to("cuda").contiguous()


def weights(case):
    return gdn.make_weights(case.conv_w, case.dt_bias, case.ssm_a, case.norm_w)


def dims(case, out_dtype=torch.float32, check_finite=False, prefill_fp32=False, state_dtype=torch.float32):
    return gdn.make_dims(case.Hk, case.Hv, case.act_dtype, out_dtype, check_finite=check_finite,
                         prefill_fp32=prefill_fp32, state_dtype=state_dtype)


def half_ulp_bf16(ref):
    a = np.abs(ref).astype(np.float32)
    e = np.floor(np.log2(np.maximum(a, 1e-30)))
    return np.where(a > 0, 2.0 ** (e - 8), 0.0)


def assert_out_close(y, ref, act_dtype, rows=None):
    """fp32 output: max |y - ref| <= tol.  bf16 output: <= tol + half a bf16 ulp of ref."""
    tol_y = TOL[act_dtype][0]
    is_bf16 = y.dtype == torch.bfloat16
    y = y.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        y = y[rows]
    assert np.all(np.isfinite(y))
    err = np.abs(y - ref)
    bound = tol_y + (half_ulp_bf16(ref) if is_bf16 else 0.0)
    worst = float(err.max()) if err.size else 0.0
    assert np.all(err <= bound), f"max |dy| = {worst:.3e} > {tol_y}"
    return worst


def assert_out_close_bf16out(y, ref, act_dtype):
    assert y.dtype == torch.bfloat16
    return assert_out_close(y, ref, act_dtype)


def state_rel_fro(S, ref):
    S = S.cpu().numpy().astype(np.float64).reshape(-1, 128 * 128)
    ref = ref.reshape(-1, 128 * 128)
    num = np.linalg.norm(S - ref, axis=1)
    den = np.maximum(np.linalg.norm(ref, axis=1), 1e-300)
    return float((num / den).max())


def assert_state_close(S, ref, act_dtype):
    r = state_rel_fro(S, ref)
    assert r <= TOL[act_dtype][1], f"state rel Frobenius {r:.3e}"
    return r


def assert_state_one_rounding(S, ref):
    """A bf16 state: every element within one bf16 rounding of the oracle,
    |S - S_ref| <= 2^-8 |S_ref| + 1e-5 max|S_ref| (half a bf16 ulp is at most
    2^-8 of the value; the second term covers the fp32 arithmetic)."""
    S = S.float().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref, dtype=np.float64).reshape(S.shape)
    err = np.abs(S - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-5 * np.abs(ref).max()
    assert np.all(err <= bound), f"worst excess {float((err - bound).max()):.3e}"


def conv_bits_equal(conv_dev, conv_ref_f32, act_dtype):
    got = conv_dev.cpu()
    want = torch.from_numpy(np.ascontiguousarray(conv_ref_f32)).to(act_dtype)
    return torch.equal(got.view(torch.int16) if act_dtype == torch.bfloat16 else got.view(torch.int32),
                       want.view(torch.int16) if act_dtype == torch.bfloat16 else want.view(torch.int32))
