"""CPU oracle of the gated DeltaNet token mixer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and the
two share no code: the oracle does its own conv, SiLU, L2 norm, gates, delta
rule and gated RMSNorm, in fp64.

Two independent restatements of the xwen CLAUDE.md page, "Architecture cheat
sheet (Qwen 3.6, ggml-org GGUF)", "Gated DeltaNet layer" paragraph:

* ``forward``       -- the recurrent (token-by-token) definition, in C
                      (``gdn_oracle.c``), fp64, OpenMP over (sequence, v-head).
* ``chunk_forward`` -- the chunked form (chunk = 64 by default) in numpy fp64,
                      derived below from the recurrence; the same page's
                      "Ground truth" list names the recurrent and chunk=64
                      forms as the two executable forms of the delta rule.

``verify_checkpoints`` gives the per-position state checkpoints used for
speculative verification (the page's "Drafting" section: verify-walk rollback
from per-position state snapshots; the NEXTN.md page's "GDN rollback").

``in_proj`` / ``out_proj`` are the projections either side of the mixer
(attn_qkv, attn_gate, ssm_alpha, ssm_beta; ssm_out) as fp64 matmuls.

Parity status of each function is stated in its docstring; every one is pinned
by ``tests/test_oracle_*.py`` against closed forms, invariants, library
routines or brute force (none is "parity unpinned").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

D = 128          # head dimension (cheat sheet: "head dims 128")
KW = 4           # conv kernel width (cheat sheet: "kernel 4")
EPS = 1e-6       # cheat sheet: "RMSNorm eps 1e-6"; the L2 clamp uses rms_norm_eps

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libgdn_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain -O2, OpenMP, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """Open a compiled oracle library (the default build, or a test variant)."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    lib.gdn_oracle_forward.restype = ctypes.c_int
    lib.gdn_oracle_forward.argtypes = [
        ctypes.c_int, P, ctypes.c_int, ctypes.c_int, ctypes.c_double,
        P, P, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_int]
    lib.gdn_oracle_max_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = load_library(build())
    return _lib



def max_threads() -> int:
    return int(_load().gdn_oracle_max_threads())


def _f32(a) -> np.ndarray:
    """Accept numpy arrays or CPU torch tensors (bf16/fp32); widen exactly."""
    if hasattr(a, "detach"):
        a = a.detach().cpu().float().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


@dataclass
class Result:
    out: np.ndarray          # [T][Hv*128] fp64, gated-normed output
    prenorm: np.ndarray      # [T][Hv*128] fp64, o before the gated norm
    S: np.ndarray            # [N][Hv][128][128] fp64, final state
    conv_state: np.ndarray   # [N][3][C] float32 (exact raw input values)
    inter: np.ndarray | None  # [T][Hv][3*128+2]: q_hat | k_hat | v | beta | g


def forward(Hk, Hv, x, z, a_raw, b_raw, conv_w, dt_bias, ssm_a, norm_w,
            conv_state, S, cu_seqlens=None, eps=EPS, want_inter=False,
            n_threads=0, lib=None) -> Result:
    """Recurrent definition, fp64 (C).  Pinned by tests/test_oracle_pins.py.

    Shapes: x [T][C] with C = 128*(2*Hk+Hv); z [T][Hv*128]; a_raw, b_raw
    [T][Hv]; conv_w [C][4]; dt_bias, ssm_a [Hv]; norm_w [128];
    conv_state [N][3][C]; S [N][Hv][128][128] (S[j][i], i the k-index);
    cu_seqlens [N+1] (default: one sequence of length T).
    Inputs are not modified; the updated states are returned.  ``lib`` selects
    another build of the same C source (used only by the mutation tests).
    """
    lib = lib if lib is not None else _load()
    x = _f32(x); z = _f32(z); a_raw = _f32(a_raw); b_raw = _f32(b_raw)
    conv_w = _f32(conv_w); dt_bias = _f32(dt_bias); ssm_a = _f32(ssm_a)
    norm_w = _f32(norm_w)
    T = x.shape[0]
    C = D * (2 * Hk + Hv)
    if cu_seqlens is None:
        cu_seqlens = [0, T]
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    N = len(cu) - 1
    cst = _f32(conv_state).reshape(N, 3, C).copy()
    St = _f64(S).reshape(N, Hv, D, D).copy()
    assert x.shape == (T, C) and z.shape == (T, Hv * D)
    assert a_raw.shape == (T, Hv) and b_raw.shape == (T, Hv)
    assert conv_w.shape == (C, KW) and cu[-1] == T
    out = np.zeros((T, Hv * D), np.float64)
    pre = np.zeros((T, Hv * D), np.float64)
    inter = np.zeros((T, Hv, 3 * D + 2), np.float64) if want_inter else None
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p) if a is not None else None
    rc = lib.gdn_oracle_forward(N, p(cu), Hk, Hv, float(eps), p(x), p(z), p(a_raw), p(b_raw),
                                p(conv_w), p(dt_bias), p(ssm_a), p(norm_w), p(cst), p(St),
                                p(out), p(pre), p(inter), int(n_threads))
    if rc != 0:
        raise ValueError("gdn_oracle_forward rejected its arguments")
    return Result(out, pre, St, cst, inter)


def verify_checkpoints(Hk, Hv, x, z, a_raw, b_raw, conv_w, dt_bias, ssm_a, norm_w,
                       conv_state, S, K, eps=EPS, n_threads=0):
    """Speculative verify over B sequences of K tokens each (x rows b*K + p).

    Returns (out [B*K][Hv*128], prenorm, S_ckpt [B][K][Hv][128][128],
    conv_ckpt [B][K][3][C]) where checkpoint p is the state after consuming
    position p (0-based).  Built by running the recurrent definition one
    position at a time and snapshotting -- checkpoint semantics from the
    xwen page's "Drafting" section (verify-walk rollback from per-position
    state planes) and the NEXTN.md page's "GDN rollback" (n_rs_seq).
    """
    x = _f32(x); z = _f32(z); a_raw = _f32(a_raw); b_raw = _f32(b_raw)
    C = D * (2 * Hk + Hv)
    B = x.shape[0] // K
    xs = x.reshape(B, K, C); zs = z.reshape(B, K, Hv * D)
    as_ = a_raw.reshape(B, K, Hv); bs = b_raw.reshape(B, K, Hv)
    cst = _f32(conv_state).reshape(B, 3, C)
    St = _f64(S).reshape(B, Hv, D, D)
    S_ck = np.zeros((B, K, Hv, D, D)); c_ck = np.zeros((B, K, 3, C), np.float32)
    out = np.zeros((B, K, Hv * D)); pre = np.zeros((B, K, Hv * D))
    for p in range(K):
        r = forward(Hk, Hv, xs[:, p], zs[:, p], as_[:, p], bs[:, p], conv_w, dt_bias, ssm_a,
                    norm_w, cst, St, cu_seqlens=np.arange(B + 1), eps=eps, n_threads=n_threads)
        cst, St = r.conv_state, r.S
        S_ck[:, p] = St; c_ck[:, p] = cst
        out[:, p] = r.out; pre[:, p] = r.prenorm
    return out.reshape(B * K, -1), pre.reshape(B * K, -1), S_ck, c_ck


# ----------------------------------------------------------------------------
# Chunked form, numpy fp64.
#
# Derivation (from the recurrence above; d = 128, chunk of n tokens,
# Gam_t = g_1 + ... + g_t inside the chunk, S0 the state entering it):
#   S_t = e^{Gam_t} S0 + sum_{r<=t} e^{Gam_t-Gam_r} d_r k_r^T
#   d_t = beta_t (v_t - e^{g_t} S_{t-1} k_t)
#       = beta_t v_t - beta_t e^{Gam_t} S0 k_t - sum_{r<t} beta_t e^{Gam_t-Gam_r}(k_t.k_r) d_r
# so (I + A) Dm = diag(beta) V - diag(beta e^Gam) K S0^T with A strictly lower,
# A[t,r] = beta_t e^{Gam_t-Gam_r} (k_t.k_r).  With Tm = (I+A)^{-1}:
#   U = Tm diag(beta) V,  W = Tm diag(beta e^Gam) K,  Dm = U - W S0^T
#   O = (diag(e^Gam) Q S0^T + (M o Q K^T) Dm) / sqrt(d),  M[t,r] = e^{Gam_t-Gam_r}, r<=t
#   S_n = e^{Gam_n} S0 + Dm^T diag(e^{Gam_n-Gam}) K
# ----------------------------------------------------------------------------

def _silu(u):
    return u / (1.0 + np.exp(-u))


def prologue(Hk, Hv, x, conv_w, conv_state, a_raw, b_raw, dt_bias, ssm_a, eps=EPS):
    """Conv, SiLU, split, clamp L2, tiling and gates for ONE sequence, numpy fp64.

    Written independently of gdn_oracle.c (vectorised over tokens).
    Returns q_hat, k_hat [T][Hv][128] (already tiled to v-heads), v [T][Hv][128],
    beta, g [T][Hv].
    """
    x = _f64(x); W = _f64(conv_w); cst = _f64(conv_state)
    T, C = x.shape
    xx = np.concatenate([cst, x], axis=0)                 # [T+3][C], position p-3 at row p
    u = sum(W[:, j][None, :] * xx[j:j + T] for j in range(KW))
    act = _silu(u)
    q = act[:, :Hk * D].reshape(T, Hk, D)
    k = act[:, Hk * D:2 * Hk * D].reshape(T, Hk, D)
    v = act[:, 2 * Hk * D:].reshape(T, Hv, D)
    q = q / np.maximum(np.linalg.norm(q, axis=-1, keepdims=True), eps)
    k = k / np.maximum(np.linalg.norm(k, axis=-1, keepdims=True), eps)
    tile = np.arange(Hv) % Hk
    q, k = q[:, tile], k[:, tile]
    ab = _f64(a_raw) + _f64(dt_bias)[None, :]
    softplus = np.logaddexp(0.0, ab)
    g = _f64(ssm_a)[None, :] * softplus
    beta = 1.0 / (1.0 + np.exp(-_f64(b_raw)))
    return q, k, v, beta, g


def chunk_delta(Q, K, V, beta, g, S0, chunk=64):
    """Chunked delta rule for one (sequence, v-head): returns (o [T][128], S_T).

    Q, K, V [T][128]; beta, g [T]; S0 [128][128] (S[j][i]).  fp64.
    Pinned against the recurrence by brute force (tests/test_oracle_chunk.py).
    """
    from scipy.linalg import solve_triangular
    S = np.array(S0, dtype=np.float64, copy=True)
    T = Q.shape[0]
    o = np.zeros((T, D))
    for c0 in range(0, T, chunk):
        c1 = min(c0 + chunk, T)
        Qc, Kc, Vc, bc, gc = Q[c0:c1], K[c0:c1], V[c0:c1], beta[c0:c1], g[c0:c1]
        n = c1 - c0
        Gam = np.cumsum(gc)
        diff = Gam[:, None] - Gam[None, :]
        strict = np.tril(np.ones((n, n), bool), -1)
        causal = np.tril(np.ones((n, n), bool), 0)
        A = bc[:, None] * np.exp(np.where(strict, diff, -np.inf)) * (Kc @ Kc.T)
        I_A = np.eye(n) + A
        U = solve_triangular(I_A, bc[:, None] * Vc, lower=True, unit_diagonal=True)
        W = solve_triangular(I_A, (bc * np.exp(Gam))[:, None] * Kc, lower=True, unit_diagonal=True)
        Dm = U - W @ S.T
        M = np.exp(np.where(causal, diff, -np.inf))
        o[c0:c1] = (np.exp(Gam)[:, None] * (Qc @ S.T) + (M * (Qc @ Kc.T)) @ Dm) / np.sqrt(D)
        S = np.exp(Gam[-1]) * S + Dm.T @ (np.exp(Gam[-1] - Gam)[:, None] * Kc)
    return o, S


def chunk_forward(Hk, Hv, x, z, a_raw, b_raw, conv_w, dt_bias, ssm_a, norm_w,
                  conv_state, S, cu_seqlens=None, eps=EPS, chunk=64) -> Result:
    """Whole layer in chunked form (numpy fp64), same contract as ``forward``."""
    x = _f64(x); z = _f64(z); a_raw = _f64(a_raw); b_raw = _f64(b_raw)
    T = x.shape[0]
    C = D * (2 * Hk + Hv)
    if cu_seqlens is None:
        cu_seqlens = [0, T]
    cu = [int(c) for c in cu_seqlens]
    N = len(cu) - 1
    cst = _f32(conv_state).reshape(N, 3, C).copy()
    St = _f64(S).reshape(N, Hv, D, D).copy()
    out = np.zeros((T, Hv * D)); pre = np.zeros((T, Hv * D))
    w = _f64(norm_w)
    for s in range(N):
        t0, t1 = cu[s], cu[s + 1]
        if t1 == t0:
            continue
        q, k, v, beta, g = prologue(Hk, Hv, x[t0:t1], conv_w, cst[s], a_raw[t0:t1],
                                    b_raw[t0:t1], dt_bias, ssm_a, eps)
        for h in range(Hv):
            o, St[s, h] = chunk_delta(q[:, h], k[:, h], v[:, h], beta[:, h], g[:, h],
                                      St[s, h], chunk)
            pre[t0:t1, h * D:(h + 1) * D] = o
            rms = np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
            zz = z[t0:t1, h * D:(h + 1) * D]
            out[t0:t1, h * D:(h + 1) * D] = o / rms * w[None, :] * _silu(zz)
        xx = np.concatenate([cst[s], _f32(x[t0:t1])], axis=0)
        cst[s] = xx[-3:]
    return Result(out, pre, St, cst, None)


def in_proj(hidden, W_qkv, W_z, W_a, W_b):
    """The projections in front of the mixer, fp64: the xwen CLAUDE.md page, "Architecture
    cheat sheet", "Gated DeltaNet layer" -- the layer input through attn_qkv (the fused q|k|v
    stream x), attn_gate (z), ssm_alpha (a_raw) and ssm_beta (b_raw).  Each weight is in the
    [out][in] layout of a linear layer, so a projection is hidden . W^T (a library matmul, the
    only step).  Returns (x, z, a_raw, b_raw).  Pinned by tests/test_oracle_pins.py (identity
    and selector weights, brute-force sums on tiny inputs)."""
    h = _f64(hidden)
    return tuple(h @ _f64(W).T for W in (W_qkv, W_z, W_a, W_b))


def out_proj(y, W_out):
    """ssm_out after the gated RMSNorm (same page and paragraph): y . W_out^T in fp64.
    Pinned with in_proj."""
    return _f64(y) @ _f64(W_out).T
