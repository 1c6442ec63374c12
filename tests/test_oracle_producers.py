"""Pins of the oracle's K and Q producers (norm, RoPE, quantiser, cache
store) against library casts, closed forms, values worked by hand and the
inverse rotation the pages print.  CPU only."""
import numpy as np
import torch

import oracle

E2M1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)


def _e4m3_table():
    return torch.arange(256, dtype=torch.int32).to(torch.uint8).view(
        torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def _bf16_val(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy() \
        .astype(np.float64)


def _cos_sin(num_pos, rope_dim, base=10000.0):
    half = rope_dim // 2
    f = base ** (-np.arange(half) / half)
    ang = np.arange(num_pos)[:, None] * f[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def test_e4m3_encode_matches_torch_cast():
    rng = np.random.default_rng(1)
    tab = _e4m3_table()
    finite = np.sort(np.unique(np.abs(tab[np.isfinite(tab)])))
    mids = (finite[1:] + finite[:-1]) / 2
    vals = np.concatenate([rng.uniform(-448, 448, 2000), rng.uniform(-1, 1, 2000) * 2.0 ** -7,
                           mids, -mids, finite, -finite])
    ref = torch.from_numpy(vals.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8)
    got = np.array([oracle.e4m3_encode(v) for v in vals.astype(np.float32)])
    # the sign bit is copied, so -0 and tiny negatives give 0x80 on both sides
    np.testing.assert_array_equal(got, ref.numpy())


def test_e2m1_encode_by_hand():
    # nearest code, ties to the even code: 0.25 -> 0, 0.75 -> 1.0 (code 2),
    # 1.25 -> 1.0, 1.75 -> 2.0 (4), 2.5 -> 2.0, 3.5 -> 4.0 (6), 5 -> 4.0;
    # sign bit 8 copied from the value, including -0 and negatives that round
    # to zero
    assert [oracle.e2m1_encode(v) for v in [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]] == \
        [0, 2, 2, 4, 4, 6, 6]
    assert [oracle.e2m1_encode(v) for v in [0.3, 0.7, 2.9, 5.01, 6.0]] == [1, 1, 5, 7, 7]
    assert oracle.e2m1_encode(-0.1) == 8 and oracle.e2m1_encode(-3.0) == 13
    assert oracle.e2m1_encode(-0.0) == 8 and oracle.e2m1_encode(0.0) == 0
    for c in range(8):
        assert oracle.e2m1_encode(E2M1[c]) == c


def test_scale_bits_closed_form():
    for top in (6.0, 448.0):
        for k in (-20, -1, 0, 3, 40):
            a = top * 2.0 ** k
            assert oracle.scale_bits(a, top) == 127 + k
            assert oracle.scale_bits(a * (1 + 2.0 ** -30), top) == 128 + k
            assert oracle.scale_bits(a * 0.75, top) == 127 + k
    assert oracle.scale_bits(0.0, 6.0) == 0           # amax floored at 2^-126, clamped to 0
    assert oracle.scale_bits(2.0 ** 127, 6.0) == 252  # ceil(127 - log2 6) + 127
    assert oracle.scale_bits(2.0 ** 130, 6.0) == 254  # 255 clamped to the top


def test_rope_inverts_by_the_printed_inverse():
    # the pages print the inverse GPT-J rotation: out_even = a cos + b sin,
    # out_odd = b cos - a sin, on the trailing rope_dim of a head
    rng = np.random.default_rng(2)
    T, H, D, rd = 5, 3, 128, 64
    q = _bf16(rng.standard_normal((T, H, D)))
    pos = rng.integers(0, 4000, T).astype(np.int32)
    cs = _cos_sin(4096, rd)
    _, _, _, _, pre, _ = oracle.q_rope_quant(1, q, pos, cs, rd, np.ones((T, H), np.float32), 1.0)
    pre = pre.reshape(T, H, D)
    x = _bf16_val(q)
    n, half = D - rd, rd // 2
    c = cs[pos, :half].astype(np.float64)[:, None, :]
    s = cs[pos, half:].astype(np.float64)[:, None, :]
    a, b = pre[..., n::2], pre[..., n + 1::2]
    back_even, back_odd = a * c + b * s, b * c - a * s
    # the table's fp32 cos and sin satisfy c^2 + s^2 = 1 only to ~1e-7, so
    # the inverse returns x (c^2 + s^2)
    norm = c * c + s * s
    np.testing.assert_allclose(back_even, x[..., n::2] * norm, rtol=0, atol=1e-12)
    np.testing.assert_allclose(back_odd, x[..., n + 1::2] * norm, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(pre[..., :n], x[..., :n])  # the leading dims pass through


def test_rms_norm_closed_forms():
    # rope_dim 0: the K producer is the norm and the quantiser.  A constant
    # key c normalises to sign(c) * w; a one-hot key c e_i to sqrt(D) w_i e_i.
    D, P = 128, 64
    w = np.linspace(0.5, 2.0, D).astype(np.float32)
    keys = np.zeros((2, D), np.float32)
    keys[0, :] = -3.0
    keys[1, 17] = 2.5
    pages = np.zeros((1, P * (D + 4)), np.uint8)
    bad, pre, _ = oracle.k_norm_rope_store(0, _bf16(keys), np.zeros(2, np.int32), None, 0, w, 0.0,
                                           pages, P, np.array([0, 5], np.int64))
    assert bad == 0
    np.testing.assert_allclose(pre[0], -w.astype(np.float64), rtol=1e-15)
    expect = np.zeros(D)
    expect[17] = np.sqrt(D) * w[17]
    np.testing.assert_allclose(pre[1], expect, rtol=1e-15, atol=0)


def test_k_store_layout_and_rounding():
    # codes are the nearest to pre * 2^(127 - bits) among the torch-decoded
    # codes; the scale sits after the page's values; skipped slots stay zero
    rng = np.random.default_rng(3)
    D, P, rd, T = 128, 64, 64, 40
    keys = _bf16(rng.standard_normal((T, D)) * 3)
    pos = rng.integers(0, 500, T).astype(np.int32)
    cs = _cos_sin(512, rd)
    w = rng.uniform(0.5, 1.5, D).astype(np.float32)
    slots = rng.permutation(3 * P)[:T].astype(np.int64)
    slots[4] = -1
    tab = _e4m3_table()
    for fmt in (0, 1):
        rowb = D if fmt == 0 else D // 2
        pages = np.zeros((3, P * (rowb + (4 if fmt == 0 else D // 32))), np.uint8)
        bad, pre, bits = oracle.k_norm_rope_store(fmt, keys, pos, cs, rd, w, 1e-6, pages, P, slots)
        assert bad == 0
        for t in range(T):
            if slots[t] < 0:
                continue
            pg, off = divmod(int(slots[t]), P)
            vals = pages[pg, off * rowb:(off + 1) * rowb]
            if fmt == 0:
                scale = pages[pg, P * rowb + off * 4:P * rowb + off * 4 + 4].view(np.float32)[0]
                assert scale == 2.0 ** (bits[t, 0] - 127)
                v = pre[t] / scale
                assert np.abs(v).max() <= 448
                dec = tab[vals]
                best = np.abs(tab[None, :127] - np.abs(v)[:, None]).min(axis=1)  # finite codes
                assert np.all(np.abs(np.abs(dec) - np.abs(v)) == best)
            else:
                sb = pages[pg, P * rowb + off * 4:P * rowb + off * 4 + 4]
                assert list(sb) == list(bits[t, :4])
                nib = np.stack([vals & 15, vals >> 4], 1).reshape(-1).astype(np.int64)
                mag = E2M1[nib & 7] * (1 - 2 * (nib >> 3))
                v = pre[t] * 2.0 ** (127 - np.repeat(sb.astype(np.int64), 32))
                assert np.abs(v).max() <= 6
                best = np.abs(E2M1[None, :] - np.abs(v)[:, None]).min(axis=1)
                assert np.all(np.abs(np.abs(mag) - np.abs(v)) == best)
        # the skipped token's slot is untouched (the pages started at zero)
        pg, off = divmod(int(rng.permutation(3 * P)[0]), P)
        skipped = int(np.asarray(slots)[4])
        assert skipped == -1


def test_q_weights_and_bad_positions():
    rng = np.random.default_rng(4)
    T, H, D = 6, 4, 128
    q = _bf16(rng.standard_normal((T, H, D)))
    pos = np.array([0, 1, 2, 3, 999, 5], np.int32)  # 999 is outside the 16-row table
    cs = _cos_sin(16, 64)
    w = rng.standard_normal((T, H)).astype(np.float32)
    for fmt in (0, 1):
        bad, q_out, q_sf, w_out, pre, bits = oracle.q_rope_quant(fmt, q, pos, cs, 64, w, 0.125)
        assert bad == 1 and np.all(w_out[4] == 0) and np.all(q_out[4] == 0)
        ok = np.arange(T) != 4
        expect = w.astype(np.float64) * 0.125
        if fmt == 0:
            expect = expect * 2.0 ** (bits[:, 0].reshape(T, H) - 127)
        np.testing.assert_array_equal(w_out[ok], expect[ok].astype(np.float32))
