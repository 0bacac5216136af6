"""The fp64 oracle against closed forms, brute force and an independent library."""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import forward as F
from oracle import stack as S

import oracle_pins as P


@pytest.mark.parametrize("check", P.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    check(F)


def test_torch_cpu_cross_check():
    """torch's CPU fp64 kernels (another code path) agree with the oracle."""
    r = np.random.default_rng(11)
    x = r.standard_normal((7, 24))
    w1, b1 = r.standard_normal((40, 24)) / 5, r.standard_normal(40) / 5
    w2, b2 = r.standard_normal((24, 40)) / 6, r.standard_normal(24) / 6
    tx = torch.from_numpy
    ref = tx(x) + torch.nn.functional.linear(
        torch.nn.functional.gelu(torch.nn.functional.linear(tx(x), tx(w1), tx(b1))), tx(w2), tx(b2))
    np.testing.assert_allclose(F.ffn_gelu(x, w1, b1, w2, b2), ref.numpy(), rtol=1e-12, atol=1e-12)
    g, u, d = r.standard_normal((40, 24)) / 5, r.standard_normal((40, 24)) / 5, r.standard_normal((24, 40)) / 6
    ref2 = tx(x) + torch.nn.functional.linear(
        torch.nn.functional.silu(torch.nn.functional.linear(tx(x), tx(g))) *
        torch.nn.functional.linear(tx(x), tx(u)), tx(d))
    np.testing.assert_allclose(F.swiglu(x, g, u, d), ref2.numpy(), rtol=1e-12, atol=1e-12)


def test_bf16_widening_exact():
    # bf16 bit patterns: 1.0 = 0x3F80, -2.5 = 0xC020, smallest normal 2^-126 = 0x0080
    bits = np.array([0x3F80, 0xC020, 0x0080, 0x0000, 0x4049], np.uint16)
    got = F.bf16_bits_to_f64(bits)
    assert got[0] == 1.0 and got[1] == -2.5 and got[2] == 2.0 ** -126 and got[3] == 0.0
    assert got[4] == 3.140625


def test_rows_are_independent():
    """The stack forward of a row subset equals those rows of the full forward
    (the sampled-row parity checks at full size rely on it)."""
    cfg = synth.TINY.with_(n_segments=3, tokens=8)
    full = S.stack_forward(cfg)
    rows = np.array([6, 1, 3])
    # equal up to BLAS blocking order (row count changes the summation blocks)
    np.testing.assert_allclose(S.stack_forward(cfg, rows=rows), full[rows], rtol=0, atol=1e-12)
    moe = synth.MOE.with_(n_segments=2, tokens=16, hidden=8, ffn=4, n_experts=6, top_k=2)
    fm = S.stack_forward(moe)
    np.testing.assert_allclose(S.stack_forward(moe, rows=np.array([15, 0, 7])), fm[[15, 0, 7]],
                               rtol=0, atol=1e-12)


def test_generator_prefix_and_determinism():
    cfg = synth.DIT
    a = synth.draw_x(cfg, tokens=16)
    b = synth.draw_x(cfg.with_(tokens=32))[:16]
    np.testing.assert_array_equal(a, b)
    t1 = synth.draw_segment(synth.TINY, 2)
    t2 = synth.draw_segment(synth.TINY, 2)
    for u, v in zip(t1, t2):
        np.testing.assert_array_equal(u, v)
    w = t1[0]
    assert w.dtype == np.float32 and w.shape == (256, 256)
    assert abs(float(w.std()) - 1 / 16) < 0.003        # N(0, 1/sqrt(256))


def test_slot_bytes_of_the_stacks():
    # aligned private footprints of the five synthetic stacks
    assert synth.segment_slot_bytes(synth.TINY) == 263_168
    assert synth.segment_slot_bytes(synth.DIT) == 16_787_456
    assert synth.segment_slot_bytes(synth.SHARED) == 151_025_664
    assert synth.segment_slot_bytes(synth.LARGE) == 424_673_280
    assert synth.segment_slot_bytes(synth.MOE) == 128 * 9_437_184
    assert sum(t.nbytes for t in synth.shared_tensors(synth.SHARED)) == 18_874_368
