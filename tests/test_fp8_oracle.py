"""Pins for the FP8 (e4m3) restatement in oracle/fp8_ref.py, checked against
the e4m3 format's definition, an independent conversion (torch's
float8_e4m3fn), the algebra of the rotation and the effect the pages print
for incoherent processing (FlashAttention-3 page, section 3)."""
import numpy as np
import pytest
import torch

from oracle import fp8_ref as f

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def test_every_e4m3_value_is_a_fixed_point():
    v = f.e4m3_values()
    assert v.size == 127 and v[0] == 0 and v[1] == 2.0 ** -9 and v[-1] == 448.0
    assert np.all(np.diff(v) > 0)
    np.testing.assert_array_equal(f.e4m3_round(v), v)
    np.testing.assert_array_equal(f.e4m3_round(-v), -v)


def test_e4m3_rounds_half_way_to_the_even_code():
    v = f.e4m3_values()
    mid = (v[:-1] + v[1:]) / 2
    got = f.e4m3_round(mid)
    codes = np.arange(v.size)
    even = np.where(codes[:-1] % 2 == 0, v[:-1], v[1:])  # code parity = mantissa parity
    np.testing.assert_array_equal(got, even)


def test_e4m3_saturates_above_448():
    np.testing.assert_array_equal(f.e4m3_round([449.0, 1e6, -500.0]), [448.0, 448.0, -448.0])


def test_e4m3_matches_an_independent_conversion():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.uniform(-448, 448, 50000), rng.standard_normal(50000) * 1e-2,
                        rng.standard_normal(20000) * 1e-3]).astype(np.float32)
    ref = torch.tensor(x).to(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(f.e4m3_round(x), ref)


def test_rotation_is_orthogonal_and_keeps_q_kt():
    rng = np.random.default_rng(4)
    signs = np.where(rng.random(128) < 0.5, -1.0, 1.0)
    m = f.rotation(signs)
    np.testing.assert_allclose(m @ m.T, np.eye(128), atol=1e-12)
    np.testing.assert_array_equal(f.hadamard(2), [[1, 1], [1, -1]])
    q, k = rng.standard_normal((7, 128)), rng.standard_normal((9, 128))
    np.testing.assert_allclose((q @ m) @ (k @ m).T, q @ k.T, atol=1e-11)


def test_block_scaling_maps_each_block_to_448():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((2, 300, 3, 128)).astype(np.float32)
    deq, codes, scales = f.quantize_row_blocks(x)
    assert scales.shape == (2, 3, 3)
    for b in range(2):
        for h in range(3):
            for t in range(3):
                assert np.abs(codes[b, t * 128:(t + 1) * 128, h]).max() == 448.0
    # relative error of a normal-range e4m3 value is at most 2^-4
    big = np.abs(x) > 0.1 * np.abs(x).max()
    assert (np.abs(deq - x)[big] <= 2.0 ** -4 * np.abs(x)[big] + 1e-9).all()


def test_rotation_reduces_fp8_error_on_outlier_inputs(oracle_mod):
    # the pages: incoherent processing cuts the FP8 attention error about 2.6x; on this
    # recipe (1 % of Q/K entries x20) require at least a 1.3x cut in O and in LSE
    from exact_attention_blackwell_gb300 import inputs

    w = inputs.Workload("o", 1, 2, 2, 512, 128, True, 2, outliers=True)
    x = inputs.make_inputs(w)
    o_ex, l_ex = oracle_mod.attention_fwd(x["q"], x["k"], x["v"], w.sm_scale, True)
    signs = np.where(np.random.default_rng(7).random(128) < 0.5, -1.0, 1.0)
    err = {}
    for name, s in (("plain", None), ("rotated", signs)):
        o, l = f.attention_fwd_fp8(x["q"], x["k"], x["v"], s, w.sm_scale, True)
        err[name] = (np.linalg.norm(o - o_ex) / np.linalg.norm(o_ex), np.sqrt(np.mean((l - l_ex) ** 2)))
    assert err["rotated"][0] * 1.3 <= err["plain"][0], err
    assert err["rotated"][1] * 1.3 <= err["plain"][1], err
