"""Python binding of libgdn.so, the GB300 (sm_103a) gated DeltaNet token mixer.

Argument marshalling only: every function below checks the tensors it is
given (device, dtype, shape, contiguity), passes their device pointers and the
current CUDA stream to the C entry point of the same name (include/gdn.h), and
raises ``GdnError`` on a non-OK status.  All arithmetic runs in the library's
CUDA kernels; there is no fallback of any kind -- without the compiled library
or a CUDA device these functions raise.

The layer is the "Gated DeltaNet layer" of the xwen CLAUDE.md page,
"Architecture cheat sheet (Qwen 3.6, ggml-org GGUF)".
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

from . import _build

__all__ = [
    "GdnError", "GdnDims", "GdnWeights", "make_dims", "make_weights", "library",
    "gdn_status_string", "gdn_version", "gdn_conv_state_init", "gdn_decode_step", "gdn_decode_step_ab",
    "gdn_verify_k", "gdn_commit", "gdn_prefill_workspace_bytes", "gdn_prefill_chunked",
    "gdn_prefill_chunked_static", "gdn_verify_k_ring", "gdn_commit_ring", "gdn_decode_step_ring",
    "gdn_state_faults", "gdn_state_reset", "GdnInProjWeights", "gdn_in_proj", "gdn_out_proj",
    "PREFILL_STATIC_SCRATCH_BYTES", "EXPORTED_SYMBOLS", "HEAD_DIM",
]

HEAD_DIM = 128
GDN_F32, GDN_BF16 = 0, 1
GDN_FLAG_CHECK_FINITE = 1
GDN_FLAG_PREFILL_FP32 = 2
GDN_FLAG_STATE_BF16 = 4
GDN_FLAG_TEST_STALL = 1 << 30
PREFILL_STATIC_SCRATCH_BYTES = 128 * 1024 * 1024   # GDN_PREFILL_STATIC_SCRATCH_BYTES

EXPORTED_SYMBOLS = (
    "gdn_status_string", "gdn_version", "gdn_conv_state_init", "gdn_decode_step", "gdn_decode_step_ab",
    "gdn_verify_k", "gdn_commit", "gdn_prefill_workspace_bytes", "gdn_prefill_chunked",
    "gdn_prefill_chunked_static", "gdn_verify_k_ring", "gdn_commit_ring", "gdn_decode_step_ring",
    "gdn_state_faults", "gdn_state_reset", "gdn_in_proj", "gdn_out_proj",
)


class GdnError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn}: {text} (status {status})")
        self.status = status


class GdnDims(ctypes.Structure):
    _fields_ = [("H_k", ctypes.c_int32), ("H_v", ctypes.c_int32), ("eps", ctypes.c_float),
                ("act_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32), ("flags", ctypes.c_uint32)]


class GdnWeights(ctypes.Structure):
    _fields_ = [("conv_w", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p), ("ssm_a", ctypes.c_void_p),
                ("norm_w", ctypes.c_void_p)]


class GdnInProjWeights(ctypes.Structure):
    _fields_ = [("W_qkv", ctypes.c_void_p), ("W_z", ctypes.c_void_p), ("W_a", ctypes.c_void_p),
                ("W_b", ctypes.c_void_p)]


_lib = None


def library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libgdn.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if build_if_missing and not _build.up_to_date():
        path = _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"libgdn.so not built ({path}); run gated_deltanet_linear_decode_gb300._build.build()")
    lib = ctypes.CDLL(path)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    D, W = ctypes.POINTER(GdnDims), ctypes.POINTER(GdnWeights)
    sig = {
        "gdn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "gdn_version": (I32, []),
        "gdn_conv_state_init": (ctypes.c_int, [D, I32, P, P, P]),
        "gdn_decode_step": (ctypes.c_int, [D, W, I32, P, P, P, P, P, P, P, P, P, P]),
        "gdn_decode_step_ab": (ctypes.c_int, [D, W, I32, I32, P, P, P, P, P, P, P, P, P, P, P]),
        "gdn_verify_k": (ctypes.c_int, [D, W, I32, I32, P, P, P, P, P, P, P, P, P, P, P, P]),
        "gdn_commit": (ctypes.c_int, [D, I32, I32, P, P, P, P, P, P]),
        "gdn_prefill_workspace_bytes": (SZ, [D, I32, ctypes.c_int64]),
        "gdn_prefill_chunked": (ctypes.c_int, [D, W, I32, P, P, P, P, P, P, P, P, I32, P, P, P, SZ, P, P]),
        "gdn_prefill_chunked_static": (ctypes.c_int, [D, W, I32, P, P, P, P, P, P, P, P, I32, P, P, P, P]),
        "gdn_verify_k_ring": (ctypes.c_int, [D, W, I32, I32, I32, P, P, P, P, P, P, P, P, P, P, P, P]),
        "gdn_commit_ring": (ctypes.c_int, [D, I32, I32, I32, P, P, P, P, P]),
        "gdn_decode_step_ring": (ctypes.c_int, [D, W, I32, I32, P, P, P, P, P, P, P, P, P, P, P]),
        "gdn_state_faults": (ctypes.c_int, [D, I32, P, I32, P, P]),
        "gdn_state_reset": (ctypes.c_int, [D, I32, I32, P, P, P, P, P]),
        "gdn_in_proj": (ctypes.c_int, [D, I32, I32, P, ctypes.POINTER(GdnInProjWeights), P, P, P, P, P, SZ, P, P]),
        "gdn_out_proj": (ctypes.c_int, [D, I32, I32, P, P, P, P, SZ, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def gdn_status_string(status: int) -> str:
    return library().gdn_status_string(int(status)).decode()


def gdn_version() -> int:
    return int(library().gdn_version())


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise GdnError(fn, status, gdn_status_string(status))


def _dt(t: torch.dtype) -> int:
    if t == torch.float32:
        return GDN_F32
    if t == torch.bfloat16:
        return GDN_BF16
    raise TypeError(f"unsupported dtype {t}")


def make_dims(Hk: int, Hv: int, act_dtype=torch.bfloat16, out_dtype=torch.float32, eps: float = 1e-6,
              check_finite: bool = False, prefill_fp32: bool = False, state_dtype=torch.float32,
              test_stall: bool = False) -> GdnDims:
    """state_dtype torch.bfloat16 selects GDN_FLAG_STATE_BF16 (bf16 activations only);
    test_stall selects GDN_FLAG_TEST_STALL (the give-up path of the kernels' waits)."""
    if state_dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("state_dtype must be torch.float32 or torch.bfloat16")
    flags = (GDN_FLAG_CHECK_FINITE if check_finite else 0) | (GDN_FLAG_PREFILL_FP32 if prefill_fp32 else 0)
    flags |= GDN_FLAG_STATE_BF16 if state_dtype == torch.bfloat16 else 0
    flags |= GDN_FLAG_TEST_STALL if test_stall else 0
    return GdnDims(Hk, Hv, eps, _dt(act_dtype), _dt(out_dtype), flags)


@dataclass
class Weights:
    conv_w: torch.Tensor   # [C][4] fp32
    dt_bias: torch.Tensor  # [H_v] fp32
    ssm_a: torch.Tensor    # [H_v] fp32
    norm_w: torch.Tensor   # [128] fp32

    def struct(self) -> GdnWeights:
        for t in (self.conv_w, self.dt_bias, self.ssm_a, self.norm_w):
            _need(t, torch.float32)
        return GdnWeights(self.conv_w.data_ptr(), self.dt_bias.data_ptr(), self.ssm_a.data_ptr(),
                          self.norm_w.data_ptr())


def make_weights(conv_w, dt_bias, ssm_a, norm_w, device="cuda") -> Weights:
    f = lambda t: t.to(device=device, dtype=torch.float32).contiguous()
    return Weights(f(conv_w), f(dt_bias), f(ssm_a), f(norm_w))


def _need(t: torch.Tensor | None, dtype=None, shape=None, optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError("missing tensor")
    if not t.is_cuda:
        raise ValueError("tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"expected shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _act(d: GdnDims):
    return torch.bfloat16 if d.act_dtype == GDN_BF16 else torch.float32


def _st(d: GdnDims):
    return torch.bfloat16 if d.flags & GDN_FLAG_STATE_BF16 else torch.float32


def _out(d: GdnDims):
    return torch.bfloat16 if d.out_dtype == GDN_BF16 else torch.float32


def gdn_conv_state_init(dims: GdnDims, conv_state: torch.Tensor, prefix: torch.Tensor | None = None,
                        stream=None) -> None:
    """conv_state [N][3][C] <- prefix (same shape) or zeros."""
    C = HEAD_DIM * (2 * dims.H_k + dims.H_v)
    N = conv_state.shape[0]
    _need(conv_state, _act(dims), (N, 3, C))
    _need(prefix, _act(dims), (N, 3, C), optional=True)
    _check("gdn_conv_state_init",
           library().gdn_conv_state_init(ctypes.byref(dims), N, _ptr(conv_state), _ptr(prefix), _stream(stream)))


def gdn_decode_step(dims: GdnDims, w: Weights, x, z, a_raw, b_raw, conv_state, S, out,
                    prenorm_out=None, dev_status=None, stream=None) -> None:
    """One recurrent step for B sequences (x [B][C]); conv_state and S in place."""
    B = x.shape[0]
    C, HvD = HEAD_DIM * (2 * dims.H_k + dims.H_v), dims.H_v * HEAD_DIM
    a = _act(dims)
    _need(x, a, (B, C)); _need(z, a, (B, HvD)); _need(a_raw, a, (B, dims.H_v)); _need(b_raw, a, (B, dims.H_v))
    _need(conv_state, a, (B, 3, C)); _need(S, _st(dims), (B, dims.H_v, HEAD_DIM, HEAD_DIM))
    _need(out, _out(dims), (B, HvD)); _need(prenorm_out, torch.float32, (B, HvD), optional=True)
    _need(dev_status, torch.int32, (B * dims.H_v,), optional=True)
    _check("gdn_decode_step", library().gdn_decode_step(
        ctypes.byref(dims), ctypes.byref(w.struct()), B, _ptr(x), _ptr(z), _ptr(a_raw), _ptr(b_raw),
        _ptr(conv_state), _ptr(S), _ptr(out), _ptr(prenorm_out), _ptr(dev_status), _stream(stream)))


def gdn_decode_step_ab(dims: GdnDims, w: Weights, x, z, hidden, W_a, W_b, conv_state, S, out,
                       prenorm_out=None, dev_status=None, stream=None) -> None:
    """gdn_decode_step with ssm_alpha / ssm_beta folded in: a_raw, b_raw formed in the kernel from
    hidden [B][H] and W_a, W_b [H_v][H] (bf16)."""
    B, H = hidden.shape
    C, HvD = HEAD_DIM * (2 * dims.H_k + dims.H_v), dims.H_v * HEAD_DIM
    a, bf = _act(dims), torch.bfloat16
    _need(x, a, (B, C)); _need(z, a, (B, HvD)); _need(hidden, bf, (B, H))
    _need(W_a, bf, (dims.H_v, H)); _need(W_b, bf, (dims.H_v, H))
    _need(conv_state, a, (B, 3, C)); _need(S, _st(dims), (B, dims.H_v, HEAD_DIM, HEAD_DIM))
    _need(out, _out(dims), (B, HvD)); _need(prenorm_out, torch.float32, (B, HvD), optional=True)
    _need(dev_status, torch.int32, (B * dims.H_v,), optional=True)
    _check("gdn_decode_step_ab", library().gdn_decode_step_ab(
        ctypes.byref(dims), ctypes.byref(w.struct()), B, H, _ptr(x), _ptr(z), _ptr(hidden), _ptr(W_a), _ptr(W_b),
        _ptr(conv_state), _ptr(S), _ptr(out), _ptr(prenorm_out), _ptr(dev_status), _stream(stream)))


def gdn_verify_k(dims: GdnDims, w: Weights, K: int, x, z, a_raw, b_raw, conv_state, S, conv_ckpt, S_ckpt,
                 out, prenorm_out=None, dev_status=None, stream=None) -> None:
    """Verify walk over K tokens per sequence (x [B*K][C]); writes per-position checkpoints."""
    B = conv_state.shape[0]
    C, HvD = HEAD_DIM * (2 * dims.H_k + dims.H_v), dims.H_v * HEAD_DIM
    a = _act(dims)
    _need(x, a, (B * K, C)); _need(z, a, (B * K, HvD)); _need(a_raw, a, (B * K, dims.H_v))
    _need(b_raw, a, (B * K, dims.H_v)); _need(conv_state, a, (B, 3, C))
    _need(S, _st(dims), (B, dims.H_v, HEAD_DIM, HEAD_DIM)); _need(conv_ckpt, a, (B, K, 3, C))
    _need(S_ckpt, _st(dims), (B, K, dims.H_v, HEAD_DIM, HEAD_DIM)); _need(out, _out(dims), (B * K, HvD))
    _need(prenorm_out, torch.float32, (B * K, HvD), optional=True)
    _need(dev_status, torch.int32, (B * dims.H_v,), optional=True)
    _check("gdn_verify_k", library().gdn_verify_k(
        ctypes.byref(dims), ctypes.byref(w.struct()), B, K, _ptr(x), _ptr(z), _ptr(a_raw), _ptr(b_raw),
        _ptr(conv_state), _ptr(S), _ptr(conv_ckpt), _ptr(S_ckpt), _ptr(out), _ptr(prenorm_out),
        _ptr(dev_status), _stream(stream)))


def gdn_commit(dims: GdnDims, K: int, accept_len, conv_ckpt, S_ckpt, conv_state, S, stream=None) -> None:
    """Make checkpoint accept_len[b]-1 the live state of every sequence b."""
    B = conv_state.shape[0]
    C = HEAD_DIM * (2 * dims.H_k + dims.H_v)
    a = _act(dims)
    _need(accept_len, torch.int32, (B,)); _need(conv_ckpt, a, (B, K, 3, C))
    _need(S_ckpt, _st(dims), (B, K, dims.H_v, HEAD_DIM, HEAD_DIM)); _need(conv_state, a, (B, 3, C))
    _need(S, _st(dims), (B, dims.H_v, HEAD_DIM, HEAD_DIM))
    _check("gdn_commit", library().gdn_commit(
        ctypes.byref(dims), B, K, _ptr(accept_len), _ptr(conv_ckpt), _ptr(S_ckpt), _ptr(conv_state), _ptr(S),
        _stream(stream)))


def gdn_verify_k_ring(dims: GdnDims, w: Weights, K: int, x, z, a_raw, b_raw, conv_state, S_ring, ring_cur,
                      conv_ckpt, out, prenorm_out=None, dev_status=None, stream=None) -> None:
    """Verify walk on the live slots of a state ring S_ring [B][R][H_v][128][128]; checkpoint p goes to
    slot (ring_cur[b] + 1 + p) % R."""
    B, R = S_ring.shape[0], S_ring.shape[1]
    C, HvD = HEAD_DIM * (2 * dims.H_k + dims.H_v), dims.H_v * HEAD_DIM
    a = _act(dims)
    _need(x, a, (B * K, C)); _need(z, a, (B * K, HvD)); _need(a_raw, a, (B * K, dims.H_v))
    _need(b_raw, a, (B * K, dims.H_v)); _need(conv_state, a, (B, 3, C))
    _need(S_ring, _st(dims), (B, R, dims.H_v, HEAD_DIM, HEAD_DIM)); _need(ring_cur, torch.int32, (B,))
    _need(conv_ckpt, a, (B, K, 3, C)); _need(out, _out(dims), (B * K, HvD))
    _need(prenorm_out, torch.float32, (B * K, HvD), optional=True)
    _need(dev_status, torch.int32, (B * dims.H_v,), optional=True)
    _check("gdn_verify_k_ring", library().gdn_verify_k_ring(
        ctypes.byref(dims), ctypes.byref(w.struct()), B, K, R, _ptr(x), _ptr(z), _ptr(a_raw), _ptr(b_raw),
        _ptr(conv_state), _ptr(S_ring), _ptr(ring_cur), _ptr(conv_ckpt), _ptr(out), _ptr(prenorm_out),
        _ptr(dev_status), _stream(stream)))


def gdn_commit_ring(dims: GdnDims, K: int, R: int, accept_len, conv_ckpt, conv_state, ring_cur, stream=None) -> None:
    """Make checkpoint accept_len[b]-1 of a ring verify the live state (slot index and conv rows only)."""
    B = conv_state.shape[0]
    C = HEAD_DIM * (2 * dims.H_k + dims.H_v)
    a = _act(dims)
    _need(accept_len, torch.int32, (B,)); _need(conv_ckpt, a, (B, K, 3, C)); _need(conv_state, a, (B, 3, C))
    _need(ring_cur, torch.int32, (B,))
    _check("gdn_commit_ring", library().gdn_commit_ring(
        ctypes.byref(dims), B, K, R, _ptr(accept_len), _ptr(conv_ckpt), _ptr(conv_state), _ptr(ring_cur),
        _stream(stream)))


def gdn_decode_step_ring(dims: GdnDims, w: Weights, x, z, a_raw, b_raw, conv_state, S_ring, ring_cur, out,
                         prenorm_out=None, dev_status=None, stream=None) -> None:
    """One recurrent step on the live slot of each sequence of a state ring, in place."""
    B, R = S_ring.shape[0], S_ring.shape[1]
    C, HvD = HEAD_DIM * (2 * dims.H_k + dims.H_v), dims.H_v * HEAD_DIM
    a = _act(dims)
    _need(x, a, (B, C)); _need(z, a, (B, HvD)); _need(a_raw, a, (B, dims.H_v)); _need(b_raw, a, (B, dims.H_v))
    _need(conv_state, a, (B, 3, C)); _need(S_ring, _st(dims), (B, R, dims.H_v, HEAD_DIM, HEAD_DIM))
    _need(ring_cur, torch.int32, (B,)); _need(out, _out(dims), (B, HvD))
    _need(prenorm_out, torch.float32, (B, HvD), optional=True)
    _need(dev_status, torch.int32, (B * dims.H_v,), optional=True)
    _check("gdn_decode_step_ring", library().gdn_decode_step_ring(
        ctypes.byref(dims), ctypes.byref(w.struct()), B, R, _ptr(x), _ptr(z), _ptr(a_raw), _ptr(b_raw),
        _ptr(conv_state), _ptr(S_ring), _ptr(ring_cur), _ptr(out), _ptr(prenorm_out), _ptr(dev_status),
        _stream(stream)))


def gdn_state_faults(dims: GdnDims, dev_status, cap: int, report=None, stream=None):
    """Summary of the non-finite status words: int32 [2 + 2*cap] on the device holding the exact
    count of faulted (sequence, v-head) pairs, the listed count, then (n*H_v + h, bits) pairs."""
    if dev_status.numel() % dims.H_v:
        raise ValueError("dev_status must hold N*H_v words")
    _need(dev_status, torch.int32, (dev_status.numel(),))
    if report is None:
        report = torch.zeros(2 + 2 * cap, dtype=torch.int32, device=dev_status.device)
    _need(report, torch.int32, (2 + 2 * cap,))
    _check("gdn_state_faults", library().gdn_state_faults(
        ctypes.byref(dims), dev_status.numel() // dims.H_v, _ptr(dev_status), cap, _ptr(report), _stream(stream)))
    return report


def gdn_state_reset(dims: GdnDims, S, dev_status, conv_state=None, ring_cur=None, stream=None) -> None:
    """Zero the state of every faulted (sequence, v-head) -- the live ring slot when ring_cur is
    given -- and the conv rows of their sequences when conv_state is given; clear dev_status."""
    N = S.shape[0]
    R = S.shape[1] if ring_cur is not None else 0
    shape = (N, R, dims.H_v, HEAD_DIM, HEAD_DIM) if ring_cur is not None else (N, dims.H_v, HEAD_DIM, HEAD_DIM)
    _need(S, _st(dims), shape); _need(dev_status, torch.int32, (N * dims.H_v,))
    _need(ring_cur, torch.int32, (N,), optional=True)
    _need(conv_state, _act(dims), (N, 3, HEAD_DIM * (2 * dims.H_k + dims.H_v)), optional=True)
    _check("gdn_state_reset", library().gdn_state_reset(
        ctypes.byref(dims), N, R, _ptr(S), _ptr(ring_cur), _ptr(conv_state), _ptr(dev_status), _stream(stream)))


def gdn_in_proj(dims: GdnDims, hidden, W_qkv, W_z, W_a, W_b, x, z, a_raw, b_raw, workspace=None,
                dev_status=None, stream=None) -> None:
    """attn_qkv / attn_gate / ssm_alpha / ssm_beta: hidden [T][H] bf16 -> x, z, a_raw, b_raw (bf16);
    weights in the [out][in] layout (fp32 accumulation; the library's weight-streaming kernel for
    T <= 256, cuBLASLt above)."""
    T, H = hidden.shape
    C, HvD = HEAD_DIM * (2 * dims.H_k + dims.H_v), dims.H_v * HEAD_DIM
    bf = torch.bfloat16
    _need(hidden, bf, (T, H)); _need(W_qkv, bf, (C, H)); _need(W_z, bf, (HvD, H))
    _need(W_a, bf, (dims.H_v, H)); _need(W_b, bf, (dims.H_v, H))
    _need(x, bf, (T, C)); _need(z, bf, (T, HvD)); _need(a_raw, bf, (T, dims.H_v)); _need(b_raw, bf, (T, dims.H_v))
    _need(workspace, None, None, optional=True); _need(dev_status, torch.int32, (1,), optional=True)
    w = GdnInProjWeights(_ptr(W_qkv), _ptr(W_z), _ptr(W_a), _ptr(W_b))
    nws = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("gdn_in_proj", library().gdn_in_proj(ctypes.byref(dims), T, H, _ptr(hidden), ctypes.byref(w), _ptr(x),
                                                _ptr(z), _ptr(a_raw), _ptr(b_raw), _ptr(workspace), nws,
                                                _ptr(dev_status), _stream(stream)))


def gdn_out_proj(dims: GdnDims, y, W_out, out, workspace=None, dev_status=None, stream=None) -> None:
    """ssm_out: y [T][H_v*128] bf16 -> out [T][H] bf16, W_out [H][H_v*128]."""
    T, HvD = y.shape
    H = out.shape[1]
    bf = torch.bfloat16
    _need(y, bf, (T, dims.H_v * HEAD_DIM)); _need(W_out, bf, (H, HvD)); _need(out, bf, (T, H))
    _need(workspace, None, None, optional=True); _need(dev_status, torch.int32, (1,), optional=True)
    nws = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("gdn_out_proj", library().gdn_out_proj(ctypes.byref(dims), T, H, _ptr(y), _ptr(W_out), _ptr(out),
                                                  _ptr(workspace), nws, _ptr(dev_status), _stream(stream)))


def gdn_prefill_workspace_bytes(dims: GdnDims, n_seq: int, T_total: int) -> int:
    return int(library().gdn_prefill_workspace_bytes(ctypes.byref(dims), n_seq, T_total))


def gdn_prefill_chunked(dims: GdnDims, w: Weights, cu_seqlens_host, cu_seqlens_dev, x, z, a_raw, b_raw,
                        conv_state, S, out, zero_init: bool = False, prenorm_out=None, workspace=None,
                        dev_status=None, stream=None) -> None:
    """Chunked (chunk=64) prefill over packed sequences; conv_state and S in place."""
    cu = cu_seqlens_host
    if not isinstance(cu, torch.Tensor):
        cu = torch.tensor(list(cu), dtype=torch.int32)
    if cu.is_cuda or cu.dtype != torch.int32 or not cu.is_contiguous():
        raise ValueError("cu_seqlens_host must be a contiguous int32 CPU tensor")
    N = cu.numel() - 1
    T = int(cu[-1])
    C, HvD = HEAD_DIM * (2 * dims.H_k + dims.H_v), dims.H_v * HEAD_DIM
    a = _act(dims)
    _need(cu_seqlens_dev, torch.int32, (N + 1,))
    _need(x, a, (T, C)); _need(z, a, (T, HvD)); _need(a_raw, a, (T, dims.H_v)); _need(b_raw, a, (T, dims.H_v))
    _need(conv_state, a, (N, 3, C)); _need(S, _st(dims), (N, dims.H_v, HEAD_DIM, HEAD_DIM))
    _need(out, _out(dims), (T, HvD)); _need(prenorm_out, torch.float32, (T, HvD), optional=True)
    _need(dev_status, torch.int32, (N * dims.H_v,), optional=True)
    need = gdn_prefill_workspace_bytes(dims, N, T)
    ws_bytes = 0
    if workspace is not None:
        _need(workspace)
        ws_bytes = workspace.numel() * workspace.element_size()
    elif need > 0:
        raise ValueError(f"gdn_prefill_chunked needs a workspace of {need} bytes")
    _check("gdn_prefill_chunked", library().gdn_prefill_chunked(
        ctypes.byref(dims), ctypes.byref(w.struct()), N, cu.data_ptr(), _ptr(cu_seqlens_dev), _ptr(x), _ptr(z),
        _ptr(a_raw), _ptr(b_raw), _ptr(conv_state), _ptr(S), int(bool(zero_init)), _ptr(out),
        _ptr(prenorm_out), _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream)))


def gdn_prefill_chunked_static(dims: GdnDims, w: Weights, cu_seqlens_host, cu_seqlens_dev, x, z, a_raw, b_raw,
                               conv_state, S, out, zero_init: bool = False, prenorm_out=None, dev_status=None,
                               stream=None) -> None:
    """gdn_prefill_chunked without a workspace: the library's fixed device
    scratch area (PREFILL_STATIC_SCRATCH_BYTES, shared by every call) serves
    instead, for callers that cannot allocate device memory.  Problems that
    need more scratch than the area holds raise GdnError (GDN_E_WORKSPACE)."""
    cu = cu_seqlens_host
    if not isinstance(cu, torch.Tensor):
        cu = torch.tensor(list(cu), dtype=torch.int32)
    if cu.is_cuda or cu.dtype != torch.int32 or not cu.is_contiguous():
        raise ValueError("cu_seqlens_host must be a contiguous int32 CPU tensor")
    N = cu.numel() - 1
    T = int(cu[-1])
    C, HvD = HEAD_DIM * (2 * dims.H_k + dims.H_v), dims.H_v * HEAD_DIM
    a = _act(dims)
    _need(cu_seqlens_dev, torch.int32, (N + 1,))
    _need(x, a, (T, C)); _need(z, a, (T, HvD)); _need(a_raw, a, (T, dims.H_v)); _need(b_raw, a, (T, dims.H_v))
    _need(conv_state, a, (N, 3, C)); _need(S, _st(dims), (N, dims.H_v, HEAD_DIM, HEAD_DIM))
    _need(out, _out(dims), (T, HvD)); _need(prenorm_out, torch.float32, (T, HvD), optional=True)
    _need(dev_status, torch.int32, (N * dims.H_v,), optional=True)
    _check("gdn_prefill_chunked_static", library().gdn_prefill_chunked_static(
        ctypes.byref(dims), ctypes.byref(w.struct()), N, cu.data_ptr(), _ptr(cu_seqlens_dev), _ptr(x), _ptr(z),
        _ptr(a_raw), _ptr(b_raw), _ptr(conv_state), _ptr(S), int(bool(zero_init)), _ptr(out),
        _ptr(prenorm_out), _ptr(dev_status), _stream(stream)))
