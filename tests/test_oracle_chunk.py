"""Brute force on tiny inputs: the chunked (WY/UT) form of the delta rule, in
numpy fp64, equals the recurrent definition (C, fp64).  The xwen CLAUDE.md
page's "Ground truth" list names both forms (recurrent and chunk=64) as
executable forms of the same delta rule, so they must agree to rounding.

Chunk size 1 makes every chunk a single recurrence step; sizes 3 and 64 with
T not a multiple of the chunk exercise partial chunks."""
import numpy as np
import pytest

import oracle
from tests import oracle_pins as pins


def _rel(a, b):
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-300)


@pytest.mark.parametrize("chunk", [1, 3, 64])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 130])
def test_chunk_equals_recurrence(chunk, T):
    c = pins.rng_case(100 + T, Hk=2, Hv=4, T=T, s0_scale=0.05)
    rec = pins.run(oracle.forward, c)
    chk = pins.run(oracle.chunk_forward, c, chunk=chunk)
    assert _rel(chk.prenorm, rec.prenorm) < 1e-11
    assert _rel(chk.out, rec.out) < 1e-11
    assert _rel(chk.S, rec.S) < 1e-11
    assert np.array_equal(chk.conv_state, rec.conv_state)


def test_chunk_equals_recurrence_varlen():
    c = pins.rng_case(200, Hk=2, Hv=4, lengths=[70, 0, 1, 64, 129], s0_scale=0.05)
    rec = pins.run(oracle.forward, c)
    chk = pins.run(oracle.chunk_forward, c, chunk=64)
    assert _rel(chk.out, rec.out) < 1e-11 and _rel(chk.S, rec.S) < 1e-11
    assert np.array_equal(chk.conv_state, rec.conv_state)


def test_chunk_strong_decay_no_overflow():
    """ssm_a = -16 and large a_raw: cumulative gates reach ~-3000 inside a
    chunk; only differences Gam_t - Gam_r <= 0 are exponentiated, so the chunk
    form stays finite and equal to the recurrence."""
    c = pins.rng_case(201, Hk=1, Hv=2, T=130, s0_scale=0.5)
    c["ssm_a"][:] = -16.0
    c["a_raw"][:] = 3.0
    rec = pins.run(oracle.forward, c)
    chk = pins.run(oracle.chunk_forward, c, chunk=64)
    assert np.all(np.isfinite(chk.out))
    assert _rel(chk.out, rec.out) < 1e-11
