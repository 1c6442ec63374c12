"""GPU parity of the K and Q producers (through the C ABI) against the
oracle.  Quantised codes and exponents must equal the oracle's except where
the oracle's value before rounding sits within fp32-versus-fp64 rounding of
a decision boundary (a midpoint between two codes, or a block amax at a
power-of-two multiple of the element range's top); there the GPU's choice
must be one of the two neighbours.  Skipped slots stay untouched and bad
positions set the status bit."""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_indexer_mxfp4_gb300 import _binding as B

pytestmark = pytest.mark.gpu

E2M1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
E4M3 = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(
    torch.float32).numpy().astype(np.float64)
REL = 1e-5  # fp32 vs fp64 values before rounding differ by ~1e-7 relative


def _cos_sin(num_pos, rope_dim, base=10000.0):
    half = rope_dim // 2
    f = base ** (-np.arange(half) / half)
    ang = np.arange(num_pos)[:, None] * f[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def _bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16)


def _signed_codes(fmt):
    if fmt == 0:
        return np.array([E4M3[c] for c in range(256) if np.isfinite(E4M3[c])])
    return np.concatenate([E2M1, -E2M1])


def _check_block(fmt, v, gpu_vals):
    """v: oracle values after scaling (float64), gpu_vals: decoded GPU codes
    (same scale): each must be the nearest code, or a near-tie neighbour."""
    codes = _signed_codes(fmt)
    d = np.abs(codes[None, :] - v[:, None])
    best = d.min(axis=1)
    got = np.abs(gpu_vals - v)
    # in units of the scaled range (amax at 448 or 6): cancellation in the
    # rotation can leave a small value with a larger relative error
    tol = REL * np.maximum(np.abs(v), 1.0)
    assert np.all(got <= best + tol), \
        f"codes not a rounding of the oracle values: {np.max(got - best)}"
    return int(np.sum(got != best))


def _bits_ok(fmt, amax, g_bits, o_bits):
    if g_bits == o_bits:
        return True
    top = 448.0 if fmt == 0 else 6.0
    r = np.log2(max(amax, 2.0 ** -126) / top)
    return abs(r - round(r)) < REL and abs(g_bits - o_bits) == 1


def _decode(fmt, raw):
    if fmt == 0:
        return E4M3[raw]
    nib = np.stack([raw & 15, raw >> 4], -1).reshape(*raw.shape[:-1], -1).astype(np.int64)
    return E2M1[nib & 7] * (1 - 2 * (nib >> 3))


@pytest.mark.parametrize("fmt", [0, 1])
def test_k_store_matches_oracle(fmt):
    rng = np.random.default_rng(50 + fmt)
    T, D, P, rd, npages = 300, 128, 64, 64, 8
    x = (rng.standard_normal((T, D)) * rng.uniform(0.1, 10, (T, 1))).astype(np.float32)
    k_bf16 = _bf16_bits(x)
    kbits = k_bf16.view(torch.int16).numpy().view(np.uint16)
    pos = rng.integers(0, 4000, T).astype(np.int32)
    cs = _cos_sin(4096, rd)
    w = rng.uniform(0.5, 1.5, D).astype(np.float32)
    slots = rng.permutation(npages * P)[:T].astype(np.int64)
    slots[7] = -1
    rowb = D if fmt == 0 else D // 2
    sbytes = 4 if fmt == 0 else D // 32
    stride = P * (rowb + sbytes)
    ora_pages = np.zeros((npages, stride), np.uint8)
    bad, pre, obits = oracle.k_norm_rope_store(fmt, kbits, pos, cs, rd, w, 1e-6, ora_pages, P,
                                               slots)
    assert bad == 0
    pages = torch.zeros((npages, stride), dtype=torch.uint8, device="cuda")
    B.idx_get_device_status()
    B.idx_k_norm_rope_store(k_bf16.cuda(), torch.from_numpy(pos).cuda(), torch.from_numpy(cs).cuda(),
                            rd, torch.from_numpy(w).cuda(), 1e-6, pages, P,
                            torch.from_numpy(slots).cuda(), fmt)
    torch.cuda.synchronize()
    assert B.idx_get_device_status() == 0
    g = pages.cpu().numpy()
    near = 0
    for t in range(T):
        if slots[t] < 0:
            continue
        pg, off = divmod(int(slots[t]), P)
        gv = g[pg, off * rowb:(off + 1) * rowb]
        sb = g[pg, P * rowb + off * sbytes:P * rowb + (off + 1) * sbytes]
        if fmt == 0:
            gbits = [int(np.round(np.log2(sb.view(np.float32)[0]))) + 127]
        else:
            gbits = [int(b) for b in sb]
        dec = _decode(fmt, gv)
        nblk = 1 if fmt == 0 else D // 32
        span = D // nblk
        for j in range(nblk):
            seg = pre[t, j * span:(j + 1) * span]
            ob = int(obits[t, j])
            assert _bits_ok(fmt, np.abs(seg).max(), gbits[j], ob), (t, j, gbits[j], ob)
            if gbits[j] == ob:
                near += _check_block(fmt, seg * 2.0 ** (127 - ob), dec[j * span:(j + 1) * span])
    # everything outside the written slots is untouched
    written = np.zeros((npages, P), bool)
    for s in slots[slots >= 0]:
        written[s // P, s % P] = True
    for pg in range(npages):
        for off in np.nonzero(~written[pg])[0]:
            assert not g[pg, off * rowb:(off + 1) * rowb].any()
    assert near <= T * D // 1000, f"{near} codes took the other side of a near-tie"


@pytest.mark.parametrize("fmt", [0, 1])
def test_q_quant_matches_oracle(fmt):
    rng = np.random.default_rng(60 + fmt)
    T, H, D, rd = 40, 64, 128, 64
    x = (rng.standard_normal((T, H, D)) * rng.uniform(0.05, 20, (T, H, 1))).astype(np.float32)
    q_bf16 = _bf16_bits(x)
    qbits = q_bf16.view(torch.int16).numpy().view(np.uint16)
    pos = rng.integers(0, 2048, T).astype(np.int32)
    cs = _cos_sin(2048, rd)
    w = (rng.standard_normal((T, H)) / 8).astype(np.float32)
    ws = 0.088 * 0.125
    bad, o_q, o_sf, o_w, pre, obits = oracle.q_rope_quant(fmt, qbits, pos, cs, rd, w, np.float32(ws))
    assert bad == 0
    rowb = D if fmt == 0 else D // 2
    q_out = torch.zeros((T, H, rowb), dtype=torch.uint8, device="cuda")
    q_sf = torch.zeros((T, H), dtype=torch.int32, device="cuda") if fmt == 1 else None
    w_out = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    B.idx_q_rope_quant(q_bf16.cuda(), torch.from_numpy(pos).cuda(), torch.from_numpy(cs).cuda(),
                       rd, torch.from_numpy(w).cuda(), ws, fmt, q_out, w_out, q_sf)
    torch.cuda.synchronize()
    assert B.idx_get_device_status() == 0
    gq = q_out.cpu().numpy().reshape(T * H, rowb)
    gw = w_out.cpu().numpy().reshape(-1)
    gsf = None if q_sf is None else q_sf.cpu().numpy().view(np.uint8).reshape(T * H, 4)
    near = 0
    nblk = 1 if fmt == 0 else D // 32
    span = D // nblk
    for th in range(T * H):
        dec = _decode(fmt, gq[th])
        for j in range(nblk):
            seg = pre[th, j * span:(j + 1) * span]
            ob = int(obits[th, j])
            if fmt == 0:
                gb = ob if gw[th] == o_w.reshape(-1)[th] else None
            else:
                gb = int(gsf[th, j])
            if gb is None:  # FP8: the exponent shows in the weight; accept a boundary amax
                assert _bits_ok(fmt, np.abs(seg).max(), ob + 1, ob) or \
                    _bits_ok(fmt, np.abs(seg).max(), ob - 1, ob), (th, j)
                continue
            assert _bits_ok(fmt, np.abs(seg).max(), gb, ob), (th, j, gb, ob)
            if gb == ob:
                near += _check_block(fmt, seg * 2.0 ** (127 - ob), dec[j * span:(j + 1) * span])
    if fmt == 1:
        np.testing.assert_array_equal(gw, o_w.reshape(-1))  # w * scale, one fp32 rounding
    assert near <= T * H * D // 1000, f"{near} codes took the other side of a near-tie"


def test_producers_flag_bad_positions_and_slots():
    rng = np.random.default_rng(70)
    T, D, P = 4, 128, 64
    k = _bf16_bits(rng.standard_normal((T, D))).cuda()
    pos = torch.tensor([0, 1, 99, 2], dtype=torch.int32, device="cuda")   # 99: past the table
    cs = torch.from_numpy(_cos_sin(16, 64)).cuda()
    w = torch.ones(D, dtype=torch.float32, device="cuda")
    slots = torch.tensor([0, 1000, 2, 3], dtype=torch.int64, device="cuda")  # 1000: past the pool
    pages = torch.zeros((2, P * (D + 4)), dtype=torch.uint8, device="cuda")
    B.idx_get_device_status()
    B.idx_k_norm_rope_store(k, pos, cs, 64, w, 1e-6, pages, P, slots, 0)
    st = B.idx_get_device_status()
    assert st & B.DEV_BAD_PAGE and st & B.DEV_BAD_POSITION
    g = pages.cpu().numpy()
    assert g[0, 0:D].any() and g[0, 3 * D:4 * D].any() and not g[0, 2 * D:3 * D].any()
    q = _bf16_bits(rng.standard_normal((T, 2, D))).cuda()
    q_out = torch.zeros((T, 2, D), dtype=torch.uint8, device="cuda")
    w_out = torch.zeros((T, 2), dtype=torch.float32, device="cuda")
    B.idx_q_rope_quant(q, pos, cs, 64, torch.ones((T, 2), dtype=torch.float32, device="cuda"),
                       1.0, 0, q_out, w_out)
    assert B.idx_get_device_status() & B.DEV_BAD_POSITION
    assert not q_out[2].any() and q_out[3].any()
