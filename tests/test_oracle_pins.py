"""Pins of the CPU oracle against things other than itself: the OCP format
definitions (exhaustive tables and library casts), values derived on paper,
exact integer recomputation, closed forms and invariants.  CPU only."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from sparse_attention_indexer_mxfp4_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- decoders


def test_e4m3_exhaustive_matches_torch_cast():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)
    for c in range(256):
        got = oracle.e4m3_to_double(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), hex(c)
        else:
            assert got == ref[c] and math.copysign(1, got) == math.copysign(1, ref[c]), hex(c)


def test_format_points_from_spec():
    g = _golden("ocp_points.json")
    for code, val in g["e4m3"].items():
        assert oracle.e4m3_to_double(int(code, 16)) == val
    for code in g["e4m3_nan"]:
        assert math.isnan(oracle.e4m3_to_double(int(code, 16)))
    for c, val in enumerate(g["e2m1"]):
        got = oracle.e2m1_to_double(c)
        assert got == val and math.copysign(1, got) == math.copysign(1, val)
    for code, val in g["e8m0"].items():
        assert oracle.e8m0_to_double(int(code, 16)) == val
    for code in g["e8m0_nan"]:
        assert math.isnan(oracle.e8m0_to_double(int(code, 16)))


def test_e8m0_exhaustive_closed_form_and_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).to(torch.float32).numpy()
    for c in range(255):
        assert oracle.e8m0_to_double(c) == 2.0 ** (c - 127)
        if 1 <= c <= 254:  # float32 cannot hold 2^-127 as a normal; compare where it can
            assert oracle.e8m0_to_double(c) == float(ref[c])
    assert math.isnan(oracle.e8m0_to_double(255))


def test_e2m1_matches_torch_fp4_unpack():
    if not hasattr(torch, "float4_e2m1fn_x2"):
        pytest.skip("torch has no float4_e2m1fn_x2")
    # torch exposes no fp4 -> float cast on CPU in every version; the exhaustive
    # table of the OCP MX spec is the pin (test_format_points_from_spec).  Check
    # here that the sign bit is bit 3 and the magnitude grid is monotone.
    mags = [oracle.e2m1_to_double(c) for c in range(8)]
    assert mags == sorted(mags) and len(set(mags)) == 8
    assert all(oracle.e2m1_to_double(c | 8) == -oracle.e2m1_to_double(c) for c in range(8))


# --------------------------------------------------------------- tiny cases


def test_tiny_fp8_hand_derived():
    g = _golden("tiny_fp8_h2_d2.json")
    q = np.array(g["q"], np.uint8)
    k = np.array(g["k"], np.uint8)
    out = oracle.mqa_logits(synth.FMT_FP8, q, None, np.array(g["w"], np.float32), k,
                            np.array(g["k_scale"], np.float32), np.array(g["ks"]),
                            np.array(g["ke"]), g["M"], g["N"], g["H"], g["D"])
    want = np.array([[float(v) for v in row] for row in g["logits"]], np.float32)
    np.testing.assert_array_equal(out, want)


def test_tiny_mxfp4_hand_derived():
    g = _golden("tiny_mxfp4_h1_d32.json")
    q = np.zeros((1, 1, 16), np.uint8)
    q[0, 0, 0] = g["q_bytes0"]
    qs = np.array([[[g["q_scale"]]]], np.uint8)
    k = np.zeros((2, 16), np.uint8)
    k[:, 0] = g["k_bytes0"]
    ksc = np.array(g["k_scale"], np.uint8).reshape(2, 1)
    out = oracle.mqa_logits(synth.FMT_MXFP4, q, qs, np.array([[g["w"]]], np.float32), k, ksc,
                            np.array([0]), np.array([2]), 1, 2, 1, 32)
    np.testing.assert_array_equal(out[0], np.array(g["logits"], np.float32))


# ------------------------------------------------- exact integer recompute


def _e4m3_int(code):
    """e4m3 value times 2^9 as an exact integer, straight from the bit fields."""
    s, e, m = code >> 7, (code >> 3) & 15, code & 7
    mag = m if e == 0 else (8 + m) << (e - 1)
    return -mag if s else mag


def test_fp8_dot_exact_against_integer_arithmetic():
    rng = np.random.default_rng(11)
    H, D, N = 4, 128, 37
    case = synth.contiguous_case(5, 1, N, H, D, ke=[N])
    ints_q = np.vectorize(_e4m3_int)(case.q.astype(np.int64))
    ints_k = np.vectorize(_e4m3_int)(case.k.astype(np.int64))
    ones = np.ones(N, np.float32)
    for h in range(H):
        w = np.zeros((1, H), np.float32)
        w[0, h] = 1.0
        out = oracle.mqa_logits(synth.FMT_FP8, case.q, None, w, case.k, ones, case.ks,
                                case.ke, 1, N, H, D)
        for t in range(N):
            dot = int(np.dot(ints_q[0, h], ints_k[t]))  # exact, units of 2^-18
            want = np.float32(max(dot, 0) / 2.0 ** 18)
            assert out[0, t] == want, (h, t)
    assert rng is not None


def _e2m1_half_int(nib):
    mags = [0, 1, 2, 3, 4, 6, 8, 12]  # value * 2
    return -mags[nib & 7] if nib & 8 else mags[nib & 7]


def test_mxfp4_dot_exact_against_fractions():
    H, D, N = 2, 128, 9
    case = synth.contiguous_case(6, 1, N, H, D, ke=[N], fmt=synth.FMT_MXFP4)
    for h in range(H):
        w = np.zeros((1, H), np.float32)
        w[0, h] = 1.0
        out = oracle.mqa_logits(synth.FMT_MXFP4, case.q, case.q_scale, w, case.k,
                                case.k_scale, case.ks, case.ke, 1, N, H, D)
        for t in range(N):
            total = Fraction(0)
            for blk in range(D // 32):
                acc = 0
                for i in range(32 * blk, 32 * blk + 32):
                    qb, kb = case.q[0, h, i // 2], case.k[t, i // 2]
                    qn = (qb >> 4) if i % 2 else (qb & 15)
                    kn = (kb >> 4) if i % 2 else (kb & 15)
                    acc += _e2m1_half_int(int(qn)) * _e2m1_half_int(int(kn))
                e = int(case.q_scale[0, h, blk]) + int(case.k_scale[t, blk]) - 254
                total += Fraction(acc, 4) * (Fraction(2) ** e)
            want = np.float32(float(max(total, Fraction(0))))
            assert out[0, t] == want, (h, t)


# -------------------------------------------------------------- closed forms


def test_closed_form_all_ones():
    H, D, N = 3, 16, 5
    q = np.full((1, H, D), 0x38, np.uint8)  # 1.0
    k = np.full((N, D), 0x38, np.uint8)
    ks_ = np.array([0.25, 0.5, 1.0, 2.0, -1.0], np.float32)
    w = np.array([[1.0, -2.0, 0.5]], np.float32)
    out = oracle.mqa_logits(synth.FMT_FP8, q, None, w, k, ks_, [0], [N], 1, N, H, D)
    want = np.array([max(s * D, 0.0) * w.sum() for s in ks_], np.float32)
    np.testing.assert_array_equal(out[0], want)


def test_q_scale_enters_inside_relu():
    H, D, N = 2, 8, 4
    case = synth.contiguous_case(7, 2, N, H, D, ke=[N, N], with_q_scale=True)
    qs = case.q_scale.copy()
    qs[:, 1] *= -1.0
    a = oracle.mqa_logits(synth.FMT_FP8, case.q, qs, case.weights, case.k, case.k_scale,
                          case.ks, case.ke, 2, N, H, D)
    # relu(k_s * q_s * dot) with a negated q_scale equals relu(-k_s * q_s * dot):
    # flip the sign of the key scales instead and fold |q_s| into the head weights
    # of a one-head-at-a-time recomputation.
    for h in range(H):
        w = np.zeros_like(case.weights)
        w[:, h] = case.weights[:, h] * np.abs(qs[:, h])
        b = oracle.mqa_logits(synth.FMT_FP8, case.q, None, w, case.k,
                              case.k_scale * np.sign(qs[0, h]), case.ks, case.ke, 2, N, H, D)
        w2 = np.zeros_like(case.weights)
        w2[:, h] = case.weights[:, h]
        c = oracle.mqa_logits(synth.FMT_FP8, case.q, qs, w2, case.k, case.k_scale, case.ks,
                              case.ke, 2, N, H, D)
        np.testing.assert_allclose(c, b, rtol=1e-6, atol=0)
    assert np.isfinite(a).all()


# ---------------------------------------------------------------- invariants


@pytest.fixture(scope="module")
def small_case():
    return synth.contiguous_case(21, 6, 300, 8, 128, ke=[300, 299, 150, 10, 0, 300],
                                 ks=[0, 5, 0, 3, 0, 290])


def test_masked_entries_are_exactly_neg_inf(small_case):
    c = small_case
    out = oracle.mqa_logits(c.fmt, c.q, c.q_scale, c.weights, c.k, c.k_scale, c.ks, c.ke,
                            c.M, c.N, c.H, c.D)
    cols = np.arange(c.N)
    for r in range(c.M):
        inside = (cols >= c.ks[r]) & (cols < c.ke[r])
        assert np.all(np.isneginf(out[r, ~inside]))
        assert np.all(np.isfinite(out[r, inside]))


def test_relu_nonnegativity_and_linearity_in_w(small_case):
    c = small_case
    def run(w):
        return oracle.mqa_logits(c.fmt, c.q, c.q_scale, w, c.k, c.k_scale, c.ks, c.ke,
                                 c.M, c.N, c.H, c.D).astype(np.float64)
    w_pos = np.abs(c.weights)
    lp = run(w_pos)
    assert np.all(lp[np.isfinite(lp)] >= 0)
    w1, w2 = c.weights, np.roll(c.weights, 1, axis=1)
    a, b = 0.75, -1.25
    lhs = run((a * w1 + b * w2).astype(np.float32))
    with np.errstate(invalid="ignore"):
        rhs = a * run(w1) + b * run(w2)
    fin = np.isfinite(lhs)
    scale = np.abs(run(np.abs(w1))) + np.abs(run(np.abs(w2))) + 1e-30
    assert np.all(np.abs(lhs[fin] - rhs[fin]) <= 4e-7 * scale[fin])


def test_one_hot_weights_reduce_to_single_head(small_case):
    c = small_case
    h = 3
    w = np.zeros_like(c.weights)
    w[:, h] = 1.0
    full = oracle.mqa_logits(c.fmt, c.q, c.q_scale, w, c.k, c.k_scale, c.ks, c.ke,
                             c.M, c.N, c.H, c.D)
    single = oracle.mqa_logits(c.fmt, c.q[:, h:h + 1], None, np.ones((c.M, 1), np.float32),
                               c.k, c.k_scale, c.ks, c.ke, c.M, c.N, 1, c.D)
    np.testing.assert_array_equal(full, single)


def test_generator_mx_quantizer_stays_on_the_grid():
    # Data-preparation sanity: decoded MXFP4 values are within half an e2m1
    # step (times the block scale) of the drawn normals.
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, 128)).astype(np.float32)
    packed, sc = synth.mx_quantize(x)
    for r in range(0, 64, 7):
        for i in range(128):
            nib = (packed[r, i // 2] >> 4) if i % 2 else (packed[r, i // 2] & 15)
            v = oracle.e2m1_to_double(int(nib)) * oracle.e8m0_to_double(int(sc[r, i // 32]))
            step = 2.0 * oracle.e8m0_to_double(int(sc[r, i // 32]))  # widest grid gap
            assert abs(v - x[r, i]) <= step / 2 + 1e-12
