"""Pins of the 4-bit KV-cache oracle (CPU only).

The quantized cache of "Qwen3-14B Optimization", section 2.3: Lloyd-Max codebook indices,
two per byte (byte c = idx[c + 64] * 16 + idx[c]), dequantized by gather -> renormalize ->
scale -> unrotate.  The oracle's readings (codebook = 16-level Lloyd-Max levels of N(0,1);
rotation R = H D / sqrt(d); one fp32 scale per row) are pinned here to things other than
the oracle: the Lloyd-Max optimality conditions checked by independent quadrature (centroids,
midpoints, a local minimum of the distortion), the two-level closed form, scipy's Hadamard
matrix, brute-force nearest-level search, the norm and direction the dequantization must
keep, and attention over the dequantized cache recomputed with numpy.
"""
import math

import numpy as np
import pytest
import torch

import oracle

scipy_linalg = pytest.importorskip("scipy.linalg")
scipy_integrate = pytest.importorskip("scipy.integrate")

D = 128


def bf(x):
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def f64(bits):
    return torch.from_numpy(np.asarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).double().numpy()


def pdf(x):
    return math.exp(-0.5 * x * x) / math.sqrt(2 * math.pi)


def cdf(x):
    return 0.5 * math.erfc(-x / math.sqrt(2))


def rot_matrix(signs):
    return scipy_linalg.hadamard(D) @ np.diag(signs.astype(np.float64)) / math.sqrt(D)


def signs_of(seed):
    return np.where(np.random.default_rng(seed).random(D) < 0.5, -1, 1).astype(np.int8)


CODEBOOK = bf(oracle.lloyd_max(16)[0])


# ----------------------------------------------------------------------------- Lloyd-Max

def test_lloyd_max_satisfies_the_optimality_conditions():
    """Thresholds at midpoints; each level the conditional mean of its cell (computed here
    by numerical quadrature, not by the oracle's closed form); symmetric; ascending."""
    lv, thr, _ = oracle.lloyd_max(16)
    assert np.all(np.diff(lv) > 0)
    np.testing.assert_allclose(lv, -lv[::-1], atol=1e-12)
    np.testing.assert_allclose(thr, 0.5 * (lv[:-1] + lv[1:]), atol=1e-15)
    edges = [-np.inf] + list(thr) + [np.inf]
    for j in range(16):
        a, b = edges[j], edges[j + 1]
        num = scipy_integrate.quad(lambda x: x * pdf(x), a, b)[0]
        mass = scipy_integrate.quad(pdf, a, b)[0]
        assert num / mass == pytest.approx(lv[j], abs=1e-9)


def test_lloyd_max_is_a_local_minimum_of_the_distortion():
    """Moving any one level (or threshold) either way raises the mean squared error, computed
    by quadrature; the distortion itself is about 0.0095 (the 16-level Gaussian quantizer)."""
    lv, thr, _ = oracle.lloyd_max(16)

    def mse(levels, thresholds):
        edges = [-np.inf] + list(thresholds) + [np.inf]
        return sum(scipy_integrate.quad(lambda x, c=levels[j]: (x - c) ** 2 * pdf(x), edges[j], edges[j + 1])[0]
                   for j in range(16))

    base = mse(lv, thr)
    assert 0.0094 < base < 0.0096
    for j in (0, 3, 7, 12):
        for dlt in (-1e-3, 1e-3):
            l2 = lv.copy()
            l2[j] += dlt
            assert mse(l2, thr) > base
            t2 = thr.copy()
            t2[min(j, 14)] += dlt
            assert mse(lv, t2) > base


def test_two_level_quantizer_closed_form():
    """Two levels: +-sqrt(2/pi), the half-normal mean."""
    lv, thr, _ = oracle.lloyd_max(2)
    np.testing.assert_allclose(lv, [-math.sqrt(2 / math.pi), math.sqrt(2 / math.pi)], atol=1e-13)
    assert thr[0] == pytest.approx(0.0, abs=1e-15)


# ----------------------------------------------------------------------------- rotation

def test_rotation_is_the_signed_hadamard_matrix():
    sg = signs_of(1)
    x = np.random.default_rng(2).standard_normal(D)
    R = rot_matrix(sg)
    np.testing.assert_allclose(oracle.rotate(x, sg), R @ x, atol=1e-12)
    np.testing.assert_allclose(oracle.unrotate(x, sg), R.T @ x, atol=1e-12)
    np.testing.assert_allclose(oracle.unrotate(oracle.rotate(x, sg), sg), x, atol=1e-12)
    assert np.linalg.norm(oracle.rotate(x, sg)) == pytest.approx(np.linalg.norm(x), rel=1e-14)


# ----------------------------------------------------------------------------- quantizer

def unpack(packed):
    lo = packed.astype(np.int64) % 16
    hi = packed.astype(np.int64) // 16
    return np.concatenate([lo, hi])


def test_quantize_picks_the_nearest_level_and_packs_as_the_page_states():
    sg = signs_of(3)
    c = f64(CODEBOOK)
    rng = np.random.default_rng(4)
    for _ in range(20):
        x = rng.standard_normal(D) * rng.uniform(0.1, 10)
        packed, sigma = oracle.q4_quantize(x, sg, CODEBOOK)
        idx = unpack(packed)
        t = math.sqrt(D) * (rot_matrix(sg) @ x) / np.linalg.norm(x)
        want = np.argmin(np.abs(t[:, None] - c[None, :]), axis=1)
        np.testing.assert_array_equal(idx, want)
        # byte j holds idx[j + 64] * 16 + idx[j]
        np.testing.assert_array_equal(packed, (want[64:] * 16 + want[:64]).astype(np.uint8))
        assert sigma == pytest.approx(np.linalg.norm(x) / np.linalg.norm(c[want]), rel=1e-13)


def test_dequantized_row_keeps_the_norm_and_the_codeword_direction():
    """gather -> renormalize -> scale -> unrotate: ||x^|| = ||x||, and R x^ is parallel to
    c[idx]."""
    sg = signs_of(5)
    c = f64(CODEBOOK)
    x = np.random.default_rng(6).standard_normal(D) * 3.0
    packed, sigma = oracle.q4_quantize(x, sg, CODEBOOK)
    xh = oracle.q4_dequantize(packed, sigma, sg, CODEBOOK)
    assert np.linalg.norm(xh) == pytest.approx(np.linalg.norm(x), rel=1e-12)
    yh = rot_matrix(sg) @ xh
    cw = c[unpack(packed)]
    np.testing.assert_allclose(yh / np.linalg.norm(yh), cw / np.linalg.norm(cw), atol=1e-12)
    # 4 bits per coordinate: the relative error is near the quantizer's sqrt(MSE) ~ 0.1
    assert np.linalg.norm(xh - x) / np.linalg.norm(x) < 0.2


def test_dequantize_then_quantize_keeps_the_codeword_direction():
    """Re-quantizing a dequantized row gives back its scale and (its coordinates lying at
    the codebook levels, rescaled by sqrt(d) / ||c[idx]|| ~ 1) nearly all its indices."""
    sg = signs_of(7)
    rng = np.random.default_rng(8)
    x = rng.standard_normal(D)
    packed, sigma = oracle.q4_quantize(x, sg, CODEBOOK)
    xh = oracle.q4_dequantize(packed, sigma, sg, CODEBOOK)
    p2, s2 = oracle.q4_quantize(xh, sg, CODEBOOK)
    assert np.mean(unpack(p2) == unpack(packed)) > 0.9
    assert np.linalg.norm(oracle.q4_dequantize(p2, s2, sg, CODEBOOK)) == pytest.approx(np.linalg.norm(x), rel=1e-12)


def test_zero_row_dequantizes_to_zero():
    sg = signs_of(9)
    packed, sigma = oracle.q4_quantize(np.zeros(D), sg, CODEBOOK)
    assert sigma == 0.0
    np.testing.assert_array_equal(oracle.q4_dequantize(packed, sigma, sg, CODEBOOK), np.zeros(D))


# ----------------------------------------------------------------------------- decode step

def make_q4_case(B, Hq, Hkv, lens, max_seq, seed):
    rng = np.random.default_rng(seed)
    rows = B * max_seq
    g = oracle.geom(B, Hq, Hkv, D, 0, max_seq, rows)
    sg = signs_of(seed + 100)
    k_idx = np.zeros((rows, Hkv, 64), np.uint8)
    v_idx = np.zeros((rows, Hkv, 64), np.uint8)
    k_sc = np.zeros((rows, Hkv), np.float32)
    v_sc = np.zeros((rows, Hkv), np.float32)
    for r in range(rows):
        for h in range(Hkv):
            k_idx[r, h], s1 = oracle.q4_quantize(rng.standard_normal(D) * 4, sg, CODEBOOK)
            v_idx[r, h], s2 = oracle.q4_quantize(rng.standard_normal(D), sg, CODEBOOK)
            k_sc[r, h], v_sc[r, h] = s1, s2
    case = dict(g=g, q_new=bf(rng.standard_normal((B, Hq, D))), k_new=bf(rng.standard_normal((B, Hkv, D))),
                v_new=bf(rng.standard_normal((B, Hkv, D))), k_idx=k_idx, v_idx=v_idx, k_scale=k_sc, v_scale=v_sc,
                page_table=None, seq_lens=np.array(lens, np.int32), positions=np.array(lens, np.int32) - 1,
                q_norm_w=bf(1 + 0.1 * rng.standard_normal(D)), k_norm_w=bf(1 + 0.1 * rng.standard_normal(D)),
                rope_theta=1e6, eps=1e-6, signs=sg, codebook_bits=CODEBOOK)
    return case


def test_q4_step_appends_the_quantized_new_rows():
    cs = make_q4_case(2, 8, 2, [5, 9], 16, seed=10)
    r = oracle.q4_decode_step(**cs)
    assert r["status"] == 0
    kw = f64(cs["k_norm_w"])
    for b, p in enumerate(cs["positions"]):
        row = b * 16 + int(p)
        for kv in range(2):
            z = oracle.rope(oracle.rmsnorm(f64(cs["k_new"][b, kv]), kw, cs["eps"]), int(p), cs["rope_theta"])
            pk, sk = oracle.q4_quantize(z, cs["signs"], CODEBOOK)
            np.testing.assert_array_equal(r["k_idx"][row, kv], pk)
            assert r["k_scale"][row, kv] == np.float32(sk)
            pv, sv = oracle.q4_quantize(f64(cs["v_new"][b, kv]), cs["signs"], CODEBOOK)
            np.testing.assert_array_equal(r["v_idx"][row, kv], pv)
            assert r["v_scale"][row, kv] == np.float32(sv)
    # every other row untouched
    mask = np.ones(32, bool)
    mask[[0 * 16 + 4, 1 * 16 + 8]] = False
    np.testing.assert_array_equal(r["k_idx"][mask], cs["k_idx"][mask])


def test_q4_step_is_softmax_attention_over_the_dequantized_cache():
    """Attention recomputed with numpy from the dequantized rows (scipy's Hadamard for the
    unrotation), against the oracle's output."""
    cs = make_q4_case(2, 8, 2, [5, 9], 16, seed=11)
    r = oracle.q4_decode_step(**cs)
    R = rot_matrix(cs["signs"])
    c = f64(CODEBOOK)
    G = 4
    for b in range(2):
        L = int(cs["seq_lens"][b])
        for h in range(8):
            kv = h // G
            q = f64(r["q_rot"][b, h])
            K = np.stack([r["k_scale"][b * 16 + t, kv] * (R.T @ c[unpack(r["k_idx"][b * 16 + t, kv])])
                          for t in range(L)])
            V = np.stack([r["v_scale"][b * 16 + t, kv] * (R.T @ c[unpack(r["v_idx"][b * 16 + t, kv])])
                          for t in range(L)])
            s = K @ q / math.sqrt(D)
            w = np.exp(s - s.max())
            np.testing.assert_allclose(r["out"][b, h], w @ V / w.sum(), atol=1e-11)


def test_q4_attention_over_the_updated_cache_is_the_step():
    cs = make_q4_case(2, 8, 2, [5, 9], 16, seed=12)
    r = oracle.q4_decode_step(**cs)
    out = oracle.q4_attention(cs["g"], r["q_rot"], r["k_idx"], r["v_idx"], r["k_scale"], r["v_scale"], None,
                              cs["seq_lens"], cs["signs"], CODEBOOK)
    np.testing.assert_array_equal(out, r["out"])
