"""Pins of the CPU oracle against what the pages and mathematics fix.

Each test ties an oracle function to something other than itself: values
printed on the pages (tests/golden, with citations), published tables and
test vectors, closed forms, library routines (scipy, torch) or brute force.
"""
import math

import numpy as np
import pytest
import scipy.linalg
import scipy.special
import scipy.stats
import torch

import oracle as O
from conftest import golden_lines


# -- sizes, presets, seeds ([TQC] TurboQuantConfig) ----------------------------

def test_preset_compression_matches_page_table():
    """Docstring preset table: bf16 K+V bytes / slot bytes at d=128."""
    for line in golden_lines("preset_compression.txt"):
        name, printed, pinned = line.split()
        cfg = O.config_from_preset(name, 128)
        ratio = 4 * 128 / cfg.slot_size
        if int(pinned):
            assert abs(ratio - float(printed)) / float(printed) < 0.03, (name, ratio)


def test_preset_bit_widths():
    for name, want in {"turboquant_k8v4": (8, 4, False), "turboquant_4bit_nc": (4, 4, True),
                       "turboquant_k3v4_nc": (3, 4, True), "turboquant_3bit_nc": (3, 3, True)}.items():
        c = O.config_from_preset(name, 128)
        assert (c.key_quant_bits, c.value_quant_bits, c.norm_correction) == want
        assert c.seed == 42


def test_unknown_preset_lists_valid_names():
    with pytest.raises(ValueError) as e:
        O.config_from_preset("turboquant_2bit", 128)
    for name in O.PRESETS:
        assert name in str(e.value)


def test_fp8_mode_derived_fields():
    """FP8 keys: d bytes, no key MSE bits, codebook still 2**value_bits."""
    c = O.Config(head_dim=128, key_quant_bits=8, value_quant_bits=4)
    assert c.key_fp8 and c.key_mse_bits == 0 and c.mse_bits == 4 and c.n_centroids == 16
    assert c.key_packed_size == 128


@pytest.mark.parametrize("d,kb,vb,key,val,slot", [
    (128, 3, 4, 50, 68, 118),   # the k3v4 example: 48 index bytes + 2, 64 code bytes + 4
    (64, 3, 4, 26, 36, 62),
    (128, 3, 3, 50, 52, 102),
    (256, 4, 4, 130, 132, 262),
    (128, 8, 4, 128, 68, 196),
    (96, 3, 4, 38, 52, 90),     # the docstring's d=96 example
])
def test_slot_sizes(d, kb, vb, key, val, slot):
    c = O.Config(head_dim=d, key_quant_bits=kb, value_quant_bits=vb)
    assert (c.key_packed_size, c.value_packed_size, c.slot_size_aligned) == (key, val, slot)


def test_slot_size_rounds_up_to_even():
    c = O.Config(head_dim=8, key_quant_bits=3, value_quant_bits=4)  # 3+2 + 4+4 = 13
    assert c.slot_size == 13 and c.slot_size_aligned == 14


def test_layer_seed_rule():
    assert [O.layer_seed(42, l) for l in range(4)] == [42, 1379, 2716, 4053]


# -- page geometry ([PR] interface.py snippet) ------------------------------------

def test_hybrid_page_lcm():
    cfg = O.config_from_preset("turboquant_4bit_nc", 256)
    tq = O.tq_page_bytes_per_token(4, cfg.slot_size_aligned)
    skip = O.skip_page_bytes_per_token(4, 256)
    assert (tq, skip) == (1048, 4096)
    page = O.hybrid_page_bytes(tq, skip)
    assert page == 536576 and page % tq == 0 and page % skip == 0 and page // tq == 512
    # lcm, not max: max(1048, 4096) is not a multiple of 1048
    assert max(tq, skip) % tq != 0
    assert O.hybrid_page_bytes(tq, None) == tq


# -- random signs -------------------------------------------------------------

def test_splitmix64_published_vectors():
    for line in golden_lines("splitmix64_vectors.txt"):
        seed, idx, want = map(int, line.split())
        assert O.splitmix64(seed, idx + 1)[idx] == want


def test_signs_follow_top_bit():
    draws = O.splitmix64(4053, 64)
    s = O.random_signs(4053, 64)
    assert all((x >> 63 == 1) == (si < 0) for x, si in zip(draws, s))
    assert set(np.unique(s)) == {-1.0, 1.0}


# -- Walsh-Hadamard rotation ------------------------------------------------------

@pytest.mark.parametrize("d", [1, 2, 4, 16, 64, 128, 256])
def test_sylvester_matches_scipy_and_is_orthogonal(d):
    h = O.sylvester_hadamard(d)
    np.testing.assert_array_equal(h, scipy.linalg.hadamard(d))
    np.testing.assert_array_equal(h @ h.T, d * np.eye(d))


def _fwht(x):
    """Textbook in-place fast Walsh-Hadamard transform (butterflies)."""
    x = np.array(x, dtype=np.float64)
    h = 1
    while h < len(x):
        for i in range(0, len(x), 2 * h):
            a = x[i:i + h].copy()
            b = x[i + h:i + 2 * h].copy()
            x[i:i + h] = a + b
            x[i + h:i + 2 * h] = a - b
        h *= 2
    return x


def test_rotation_is_signed_hadamard():
    d = 128
    s = O.random_signs(O.layer_seed(42, 2), d)
    pi = O.rotation_matrix(s)
    np.testing.assert_allclose(pi @ pi.T, np.eye(d), atol=1e-14)
    h = scipy.linalg.hadamard(d) / math.sqrt(d)
    for j in (0, 5, 77, 127):
        np.testing.assert_allclose(pi[:, j], s[j] * h[:, j], atol=0)
    x = np.random.default_rng(0).standard_normal(d)
    np.testing.assert_allclose(pi @ x, _fwht(s * x) / math.sqrt(d), atol=1e-12)
    np.testing.assert_allclose(np.abs(pi @ np.eye(d)[0]), np.full(d, 1 / math.sqrt(d)), atol=1e-15)


# -- Lloyd-Max --------------------------------------------------------------------

def _cell_stats(edges, c):
    """Per cell: probability, first moment, second moment of N(0,1)."""
    a, b = edges[:-1], edges[1:]
    pa, pb = scipy.stats.norm.pdf(a), scipy.stats.norm.pdf(b)
    mass = scipy.stats.norm.cdf(b) - scipy.stats.norm.cdf(a)
    m1 = pa - pb
    with np.errstate(invalid="ignore"):
        ta = np.where(np.isinf(a), 0.0, a * pa)
        tb = np.where(np.isinf(b), 0.0, b * pb)
    m2 = mass + ta - tb
    return mass, m1, m2


def test_lloyd_max_fixed_point():
    for levels in (2, 4, 8, 16):
        c, _ = O.lloyd_max_normal(levels)
        edges = np.concatenate([[-np.inf], 0.5 * (c[:-1] + c[1:]), [np.inf]])
        mass, m1, _ = _cell_stats(edges, c)
        np.testing.assert_allclose(c, m1 / mass, atol=1e-12)  # centroid = cell mean
        np.testing.assert_array_equal(c, -c[::-1])            # symmetric


def test_lloyd_max_one_bit_closed_form():
    c, _ = O.lloyd_max_normal(2)
    assert abs(c[1] - math.sqrt(2 / math.pi)) < 1e-14


def test_lloyd_max_matches_max_1960_table():
    rows = {}
    for line in golden_lines("lloyd_max_normal_max1960.txt"):
        parts = line.split()
        rows[(int(parts[0]), parts[1])] = [float(x) for x in parts[2:]]
    for levels in (2, 4, 8, 16):
        c, _ = O.lloyd_max_normal(levels)
        pos = c[levels // 2:]
        want = rows[(levels, "outputs")]
        np.testing.assert_allclose(pos, want, rtol=6e-4, atol=6e-4)
        if (levels, "thresholds") in rows:
            thr = 0.5 * (pos[:-1] + pos[1:])
            np.testing.assert_allclose(thr, rows[(levels, "thresholds")], rtol=6e-4, atol=6e-4)
        edges = np.concatenate([[-np.inf], 0.5 * (c[:-1] + c[1:]), [np.inf]])
        mass, m1, m2 = _cell_stats(edges, c)
        mse = float(np.sum(m2 - 2 * c * m1 + c * c * mass))
        assert abs(mse - rows[(levels, "mse")][0]) / rows[(levels, "mse")][0] < 2e-3


def _golden_codebook_rows():
    rows = []
    for line in golden_lines("codebook_fp32_d128_b3.txt"):
        j, bits, mid, alt = (f.strip() for f in line.split("|"))
        rows.append((int(j), int(bits, 16), mid, int(alt, 16)))
    return rows


def test_codebook_boundaries_round_the_exact_midpoint():
    """fp32 boundaries are the correctly rounded exact midpoints of the scaled
    Lloyd-Max centroids (d=128, 3 bits, tests/golden/codebook_fp32_d128_b3.txt,
    derived with mpmath); the midpoint of the fp32 centroids differs."""
    cb = O.codebook(128, 3)
    got = cb.boundaries.view(np.uint32)
    c32 = cb.centroids.astype(np.float64)
    alt = (0.5 * (c32[:-1] + c32[1:])).astype(np.float32).view(np.uint32)
    differs = 0
    for j, bits, _, alt_bits in _golden_codebook_rows():
        assert got[j] == bits, (j, hex(got[j]), hex(bits))
        assert alt[j] == alt_bits, (j, hex(alt[j]), hex(alt_bits))
        differs += alt_bits != bits
    assert differs >= 1


def _rn_fp32(x, mp):
    """Correctly rounded fp32 of an mpmath value (ties to the even pattern)."""
    f = np.float32(float(x))
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    dist = [abs(mp.mpf(float(c)) - x) for c in cands]
    best = [c for c, dd in zip(cands, dist) if dd == min(dist)]
    return best[0] if len(best) == 1 else [c for c in best if int(c.view(np.uint32)) % 2 == 0][0]


@pytest.mark.parametrize("d,bits", [(64, 3), (128, 3), (128, 4), (256, 4)])
def test_codebook_tables_against_high_precision_solve(d, bits):
    """Independent 40-digit solve of the Lloyd-Max conditions for N(0,1)
    (mpmath Newton, started at Max's 1960 values): the oracle's fp32
    centroids and boundaries are its correct fp32 roundings."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    levels = 1 << bits
    half = levels // 2
    start = {8: [0.2451, 0.7560, 1.3440, 2.1520],
             16: [0.1284, 0.3881, 0.6568, 0.9424, 1.2562, 1.6181, 2.0690, 2.7326]}[levels]

    def conditions(*c):
        edges = [mp.mpf(0)] + [(c[j] + c[j + 1]) / 2 for j in range(half - 1)] + [mp.inf]
        res = []
        for j in range(half):
            a, b = edges[j], edges[j + 1]
            pb = 0 if b == mp.inf else mp.npdf(b)
            res.append(c[j] - (mp.npdf(a) - pb) / (mp.ncdf(b) - mp.ncdf(a)))
        return res

    sol = mp.findroot(conditions, [mp.mpf(x) for x in start])
    pos = [sol[i] for i in range(half)]
    sigma = 1 / mp.sqrt(d)
    pos_bnd = [sigma * (pos[j] + pos[j + 1]) / 2 for j in range(half - 1)]
    want_c = [-_rn_fp32(sigma * x, mp) for x in pos[::-1]] + [_rn_fp32(sigma * x, mp) for x in pos]
    want_b = [-_rn_fp32(x, mp) for x in pos_bnd[::-1]] + [np.float32(0.0)] + [_rn_fp32(x, mp) for x in pos_bnd]
    cb = O.codebook(d, bits)
    np.testing.assert_array_equal(cb.centroids.view(np.uint32), np.array(want_c, dtype=np.float32).view(np.uint32))
    np.testing.assert_array_equal(np.abs(cb.boundaries).view(np.uint32),
                                  np.abs(np.array(want_b, dtype=np.float32)).view(np.uint32))


def test_codebook_scaling_and_symmetry():
    for d, bits in ((64, 3), (128, 3), (128, 4), (256, 4)):
        cb = O.codebook(d, bits)
        c, _ = O.lloyd_max_normal(1 << bits)
        np.testing.assert_array_equal(cb.centroids, (c / math.sqrt(d)).astype(np.float32))
        np.testing.assert_array_equal(cb.centroids, -cb.centroids[::-1])
        np.testing.assert_array_equal(cb.boundaries, -cb.boundaries[::-1])
        assert cb.boundaries[(1 << bits) // 2 - 1] == 0.0
        assert np.all(np.diff(cb.boundaries) > 0)


@pytest.mark.parametrize("bits,mse", [(3, 0.03454), (4, 0.009497)])
def test_rotated_key_distortion_matches_gaussian_mse(bits, mse):
    """A random rotation makes a unit key's coordinates ~N(0, 1/d), so the
    quantised unit vector's squared error approaches Max's distortion."""
    d = 256
    layer = O.make_layer(O.Config(head_dim=d, key_quant_bits=bits, value_quant_bits=4), 0)
    k = np.random.default_rng(1).standard_normal((600, d))
    idx, _, _ = O.encode_keys_mse(k, layer.pi, layer.cb)
    y = (k / np.linalg.norm(k, axis=1, keepdims=True)) @ layer.pi.T
    err = np.sum((y - layer.cb.centroids[idx]) ** 2, axis=1).mean()
    assert abs(err - mse) / mse < 0.05


def test_key_index_is_nearest_centroid():
    d = 64
    layer = O.make_layer(O.Config(head_dim=d, key_quant_bits=3), 0)
    k = np.random.default_rng(2).standard_normal((300, d))
    idx, norm, near = O.encode_keys_mse(k, layer.pi, layer.cb)
    y = (k / np.linalg.norm(k, axis=1, keepdims=True)) @ layer.pi.T
    brute = np.argmin(np.abs(y[:, :, None] - layer.cb.centroids[None, None, :].astype(np.float64)), axis=2)
    assert np.all((idx == brute) | near)
    np.testing.assert_array_equal(norm, np.linalg.norm(k, axis=1).astype(np.float16))


def test_zero_key_encodes_middle_cell():
    layer = O.make_layer(O.Config(head_dim=16, key_quant_bits=4), 0)
    idx, norm, _ = O.encode_keys_mse(np.zeros((1, 16)), layer.pi, layer.cb)
    assert np.all(idx == 7) and norm[0] == 0


# -- codecs -----------------------------------------------------------------------

def test_bitpack_worked_examples():
    for line in golden_lines("bitpack_examples.txt"):
        bits, codes, hexes = (f.strip() for f in line.split("|"))
        codes = np.array([[int(x) for x in codes.split()]])
        want = np.array([[int(h, 16) for h in hexes.split()]], dtype=np.uint8)
        got = O.pack_bits(codes, int(bits))
        np.testing.assert_array_equal(got, want)
        np.testing.assert_array_equal(O.unpack_bits(got, int(bits), codes.shape[1]), codes)


def test_fp16_little_endian():
    np.testing.assert_array_equal(O.f16_bytes(np.array([1.0, -2.0], dtype=np.float16)),
                                  [[0x00, 0x3C], [0x00, 0xC0]])


def test_bf16_round_matches_torch():
    x = np.concatenate([np.random.default_rng(3).standard_normal(10000).astype(np.float32) * 37,
                        np.array([0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, 3e38, 1e-40], dtype=np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(O.bf16_round(x).view(np.uint32), want.view(np.uint32))


def _e4m3_table():
    vals = np.array([O.e4m3_value(c) for c in range(256)])
    return vals


def test_e4m3_decode_known_values():
    assert O.e4m3_value(0x38) == 1.0
    assert O.e4m3_value(0x7E) == 448.0
    assert O.e4m3_value(0x01) == 2.0 ** -9
    assert O.e4m3_value(0x08) == 2.0 ** -6
    assert O.e4m3_value(0xB8) == -1.0
    assert math.isnan(O.e4m3_value(0x7F))


def test_e4m3_encode_exhaustive_bf16_bruteforce():
    """Every finite bf16 bit pattern against a brute-force nearest search over
    the positive e4m3 codes (ties to the even code, saturating at 448); the
    sign bit is copied, so values that round to zero keep their sign."""
    bits = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        x = (bits << 16).view(np.float32).astype(np.float64)
    x = x[np.isfinite(x)]
    table = _e4m3_table()
    codes = np.arange(0x7F)  # 0x00 .. 0x7E: +0 .. 448
    vals = table[codes]
    a = np.minimum(np.abs(x), 448.0)
    dist = np.abs(a[:, None] - vals[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = np.where(dist == best, codes[None, :], 1 << 20)
    even = np.where((cand & 1) == 0, cand, 1 << 20).min(axis=1)
    brute = np.where(even < (1 << 20), even, cand.min(axis=1))
    brute = brute | np.where(np.signbit(x), 0x80, 0)
    got = O.e4m3_encode(x)
    np.testing.assert_array_equal(got, brute.astype(np.uint8))
    # torch's own e4m3fn cast agrees inside the finite range
    inr = np.abs(x) <= 448
    t = torch.from_numpy(x[inr].astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(got[inr], t)


def test_value_quant_worked_grid():
    """A vector already on an fp16 grid z0 + s0*j (s0 = range/15 exactly)
    gets codes j and reconstructs exactly."""
    z0, s0 = np.float32(-1.5), np.float32(0.25)
    v = (z0 + s0 * np.arange(16, dtype=np.float32))[None, :].repeat(2, 0)
    v[1] = v[1][::-1]
    codes, scale, zero = O.encode_values(v, 4)
    np.testing.assert_array_equal(codes[0], np.arange(16))
    np.testing.assert_array_equal(codes[1], np.arange(16)[::-1])
    assert scale[0] == np.float16(0.25) and zero[0] == np.float16(-1.5)


def test_value_quant_constant_vector():
    v = np.full((1, 32), 0.3, dtype=np.float32)
    codes, scale, zero = O.encode_values(v, 3)
    assert scale[0] == 0 and np.all(codes == 0) and zero[0] == np.float16(0.3)


@pytest.mark.parametrize("bits", [3, 4])
def test_value_quant_error_bound(bits):
    v = O.bf16_round(np.random.default_rng(4).standard_normal((500, 128)).astype(np.float32) * 3)
    codes, scale, zero = O.encode_values(v, bits)
    top = (1 << bits) - 1
    assert codes.min() >= 0 and codes.max() <= top
    s = scale.astype(np.float64)[:, None]
    z = zero.astype(np.float64)[:, None]
    v_hat = s * codes + z
    slack = 2.0 ** -10 * np.abs(v).max(axis=1, keepdims=True) * (top + 1)
    assert np.all(np.abs(v_hat - v) <= 0.5 * s + slack)
    # most vectors use both ends of the code range
    assert np.mean(codes.min(axis=1) == 0) > 0.9 and np.mean(codes.max(axis=1) == top) > 0.9


def test_value_quant_readings_hand_worked():
    """tests/golden/value_quant_readings.txt: codes decided against the fp16
    scale and zero a reader sees, ties to even; each row also fails the
    rejected reading it names."""
    for line in golden_lines("value_quant_readings.txt"):
        bits, vals, sbits, zbits, codes, rejected, _ = (f.strip() for f in line.split("|"))
        v = np.array([[float(x) for x in vals.split()]], dtype=np.float32)
        got_codes, scale, zero = O.encode_values(v, int(bits))
        assert int(scale.view(np.uint16)[0]) == int(sbits, 16)
        assert int(zero.view(np.uint16)[0]) == int(zbits, 16)
        want = [int(x) for x in codes.split()]
        np.testing.assert_array_equal(got_codes[0], want)
        assert want != [int(x) for x in rejected.split()]


# -- slots, cache and dequant -------------------------------------------------------

def test_slot_layout_fp8_fields():
    cfg = O.Config(head_dim=16, key_quant_bits=8, value_quant_bits=4)
    layer = O.make_layer(cfg, 0)
    k = np.linspace(-2, 2, 16)[None]
    v = np.arange(16, dtype=np.float64)[None] * 0.5
    slot, _ = O.encode_slots(layer, k, v)
    assert slot.shape == (1, 16 + 8 + 4)
    np.testing.assert_array_equal(slot[0, :16], O.e4m3_encode(k[0]))
    assert O.f16_from_bytes(slot[:, 24:26])[0] == 0.5 and O.f16_from_bytes(slot[:, 26:28])[0] == 0.0
    np.testing.assert_array_equal(O.unpack_bits(slot[:, 16:24], 4, 16)[0], np.arange(16))


def test_cache_scatter_roundtrip():
    cfg = O.Config(head_dim=16, key_quant_bits=3, value_quant_bits=3)
    layer = O.make_layer(cfg, 1)
    rng = np.random.default_rng(5)
    k = O.bf16_round(rng.standard_normal((40, 2, 16)).astype(np.float32))
    v = O.bf16_round(rng.standard_normal((40, 2, 16)).astype(np.float32))
    cache = O.new_cache(cfg, 6, 8, 2, block_stride=8 * 2 * cfg.slot_size_aligned + 16)
    table = np.array([[4, 1, 5, 0, 2]])
    slots = table[0, np.arange(40) // 8] * 8 + np.arange(40) % 8
    slots[7] = -1
    O.store_kv(layer, k, v, slots, cache)
    got = np.stack([O.read_slots(cache, table[0], 40, h) for h in range(2)], axis=1)
    want, _ = O.encode_slots(layer, k.reshape(-1, 16), v.reshape(-1, 16))
    want = want.reshape(40, 2, -1)
    keep = np.arange(40) != 7
    np.testing.assert_array_equal(got[keep], want[keep])
    assert np.all(got[7] == 0)
    # the same bytes at addresses worked out by hand: block table[t // 8] at
    # its (padded) stride, then position t % 8 and head h in [B, H, slot] order
    sb = cfg.slot_size_aligned
    for t in np.flatnonzero(keep):
        for h in range(2):
            off = table[0, t // 8] * cache.block_stride + ((t % 8) * 2 + h) * sb
            np.testing.assert_array_equal(cache.data[off:off + sb], want[t, h])


def test_dequant_reconstruction_and_nc():
    d = 128
    rng = np.random.default_rng(6)
    k = O.bf16_round(rng.standard_normal((200, d)).astype(np.float32))
    v = O.bf16_round(rng.standard_normal((200, d)).astype(np.float32))
    plain = O.make_layer(O.Config(head_dim=d, key_quant_bits=4, value_quant_bits=4), 3)
    nc = O.make_layer(O.Config(head_dim=d, key_quant_bits=4, value_quant_bits=4, norm_correction=True), 3)
    slots, _ = O.encode_slots(plain, k, v)
    kp, vp = O.dequant_slots(plain, slots)
    kn, vn = O.dequant_slots(nc, slots)
    # NC only renormalises the centroid vector: ||k_hat|| = vec_norm exactly
    np.testing.assert_allclose(np.linalg.norm(kn, axis=1),
                               np.linalg.norm(k, axis=1).astype(np.float16).astype(np.float64), rtol=1e-12)
    ratio = np.linalg.norm(kn, axis=1) / np.linalg.norm(kp, axis=1)
    np.testing.assert_allclose(kn, kp * ratio[:, None], rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(vp, vn)
    # reconstruction quality: relative error near the 4-bit distortion
    rel = np.sum((kp - k) ** 2, axis=1) / np.sum(k * k, axis=1)
    assert rel.mean() < 0.015


def test_dequant_cache_varlen_layout_from_hand_built_slots():
    """dequant_cache against slots written byte by byte: FP8 keys decoded by
    torch's float8_e4m3fn, values fp32(scale) * code + fp32(zero) with one
    fp32 rounding (the product is exact) and torch's bf16 rounding, and token
    j of sequence s in row cu_seqlens[s] + j through a permuted block table
    and a padded block stride."""
    import torch

    d, h_n, bs = 16, 2, 4
    cfg = O.Config(head_dim=d, key_quant_bits=8, value_quant_bits=4)
    layer = O.make_layer(cfg, 0)
    slot_bytes = 16 + 8 + 4
    assert cfg.slot_size_aligned == slot_bytes
    stride = bs * h_n * slot_bytes + 32
    cache = O.new_cache(cfg, 8, bs, h_n, block_stride=stride)
    lens = [5, 11]
    table = np.array([[6, 1, 0, 0], [3, 7, 0, 5]])
    cu = np.array([0, 5, 16])
    s16, z16 = np.float16(0.1), np.float16(0.3)
    want_k = np.zeros((16, h_n, d), dtype=np.float32)
    want_v = np.zeros((16, h_n, d), dtype=np.float32)
    for s, n in enumerate(lens):
        for j in range(n):
            for h in range(h_n):
                row = cu[s] + j
                kb = np.array([(7 * row + 5 * h + 3 * i) % 0x77 for i in range(d)], dtype=np.uint8)
                codes = np.array([(row + 3 * h + i) % 16 for i in range(d)])
                packed = np.array([codes[2 * b] | (codes[2 * b + 1] << 4) for b in range(d // 2)], dtype=np.uint8)
                tail = np.frombuffer(np.array([s16, z16], dtype="<f2").tobytes(), dtype=np.uint8)
                off = table[s, j // bs] * stride + ((j % bs) * h_n + h) * slot_bytes
                cache.data[off:off + slot_bytes] = np.concatenate([kb, packed, tail])
                want_k[row, h] = torch.from_numpy(kb).view(torch.float8_e4m3fn).float().numpy()
                exact32 = np.float32(s16) * codes.astype(np.float32) + np.float32(z16)
                want_v[row, h] = torch.from_numpy(exact32).to(torch.bfloat16).float().numpy()
    k_out, v_out = O.dequant_cache(layer, cache, table, cu)
    np.testing.assert_array_equal(k_out, want_k)
    np.testing.assert_array_equal(v_out, want_v)


# -- decode ---------------------------------------------------------------------

def _tiny_cache(layer, n_tok, h_n, k, v):
    cfg = layer.cfg
    bs = 16
    nblk = (n_tok + bs - 1) // bs
    cache = O.new_cache(cfg, nblk, bs, h_n)
    table = np.arange(nblk)[::-1].copy()[None]
    slots = table[0, np.arange(n_tok) // bs] * bs + np.arange(n_tok) % bs
    O.store_kv(layer, k, v, slots, cache)
    return cache, table


def test_decode_matches_scipy_softmax_on_dequantised_cache():
    cfg = O.Config(head_dim=32, key_quant_bits=3, value_quant_bits=4, norm_correction=True)
    layer = O.make_layer(cfg, 0)
    rng = np.random.default_rng(7)
    k = O.bf16_round(rng.standard_normal((37, 2, 32)).astype(np.float32))
    v = O.bf16_round(rng.standard_normal((37, 2, 32)).astype(np.float32))
    q = O.bf16_round(rng.standard_normal((1, 4, 32)).astype(np.float32))
    cache, table = _tiny_cache(layer, 37, 2, k, v)
    out = O.decode_attention(layer, q, cache, table, np.array([37]))
    for hq in range(4):
        h = hq // 2
        sl = O.read_slots(cache, table[0], 37, h)
        kh, vh = O.dequant_slots(layer, sl)
        p = scipy.special.softmax(kh @ q[0, hq].astype(np.float64) / math.sqrt(32))
        np.testing.assert_allclose(out[0, hq], p @ vh, rtol=1e-12, atol=1e-12)
        # the fused form: q . k_hat = vec_norm * (Pi q) . c~ / ||c~||
        nb = cfg.key_packed_size - 2
        idx = O.unpack_bits(sl[:, :nb], 3, 32)
        c = layer.cb.centroids.astype(np.float64)[idx]
        n = O.f16_from_bytes(sl[:, nb:nb + 2])
        fused = n * (c @ (layer.pi @ q[0, hq].astype(np.float64))) / np.linalg.norm(c, axis=1)
        np.testing.assert_allclose(kh @ q[0, hq].astype(np.float64), fused, rtol=1e-11, atol=1e-12)


def test_decode_special_cases():
    cfg = O.Config(head_dim=16, key_quant_bits=4, value_quant_bits=3)
    layer = O.make_layer(cfg, 0)
    rng = np.random.default_rng(8)
    k = O.bf16_round(rng.standard_normal((20, 1, 16)).astype(np.float32))
    v = O.bf16_round(rng.standard_normal((20, 1, 16)).astype(np.float32))
    cache, table = _tiny_cache(layer, 20, 1, k, v)
    q = O.bf16_round(rng.standard_normal((1, 1, 16)).astype(np.float32))
    _, vh = O.dequant_slots(layer, O.read_slots(cache, table[0], 20, 0))
    # a single cached token: the output is its value
    np.testing.assert_array_equal(O.decode_attention(layer, q, cache, table, np.array([1]))[0, 0], vh[0])
    # a zero query weights every token equally
    np.testing.assert_allclose(O.decode_attention(layer, np.zeros_like(q), cache, table, np.array([20]))[0, 0],
                               vh.mean(axis=0), rtol=1e-13, atol=1e-14)
    # no cached tokens: zero row
    assert np.all(O.decode_attention(layer, q, cache, table, np.array([0])) == 0)
    # identical keys: mean of the values
    same = np.repeat(k[:1], 20, axis=0)
    cache2, table2 = _tiny_cache(layer, 20, 1, same, v)
    np.testing.assert_allclose(O.decode_attention(layer, q, cache2, table2, np.array([20]))[0, 0],
                               vh.mean(axis=0), rtol=1e-12, atol=1e-13)


def test_split_merge_is_exact():
    rng = np.random.default_rng(9)
    kh = rng.standard_normal((101, 16))
    vh = rng.standard_normal((101, 16))
    q = rng.standard_normal(16) * 3
    full = O.attention_row(q, kh, vh, 0.25)
    for cuts in ([50], [1, 2, 3, 99], list(range(7, 101, 7))):
        edges = [0, *cuts, 101]
        parts = [O.partial_state(q, kh[a:b], vh[a:b], 0.25) for a, b in zip(edges[:-1], edges[1:])]
        np.testing.assert_allclose(O.merge_partials(parts), full, rtol=1e-12, atol=1e-13)


# ---- ring-buffered store ([ART] article, full_tq write path) ---------------------------

def _ring_inputs(rng, lens, h_n, d):
    k = [O.bf16_round(rng.standard_normal((n, h_n, d)).astype(np.float32)) for n in lens]
    v = [O.bf16_round(rng.standard_normal((n, h_n, d)).astype(np.float32)) for n in lens]
    return k, v


def _ring_setup(layer, lens, h_n, r_len, block_size=16):
    nblk = [max(1, -(-n // block_size)) for n in lens]
    table = np.zeros((len(lens), max(nblk)), dtype=np.int64)
    perm = np.random.default_rng(11).permutation(sum(nblk))
    off = 0
    for s, nb in enumerate(nblk):
        table[s, :nb] = perm[off:off + nb]
        off += nb
    cache = O.new_cache(layer.cfg, sum(nblk), block_size, h_n)
    d = layer.cfg.head_dim
    ring_k = np.zeros((len(lens), r_len, h_n, d), dtype=np.float32)
    return cache, table, ring_k, ring_k.copy()


def test_ring_steps_pack_exactly_the_whole_blocks():
    """Token-by-token appends leave the same packed bytes as one plain store
    of every whole ring block, and the remainder verbatim in the ring."""
    cfg = O.Config(head_dim=16, key_quant_bits=3, value_quant_bits=4, norm_correction=True)
    layer = O.make_layer(cfg, 0)
    lens, r_len, h_n = [70, 33, 32], 32, 2
    k, v = _ring_inputs(np.random.default_rng(21), lens, h_n, 16)
    cache, table, ring_k, ring_v = _ring_setup(layer, lens, h_n, r_len)
    for step in range(max(lens)):
        cur = np.array([step if step < n else -1 for n in lens])
        ks = np.stack([k[s][min(step, n - 1)] for s, n in enumerate(lens)])
        vs = np.stack([v[s][min(step, n - 1)] for s, n in enumerate(lens)])
        O.ring_append(layer, cache, table, ring_k, ring_v, cur, ks, vs, np.arange(len(lens) + 1))
    want = O.new_cache(cfg, cache.num_blocks, cache.block_size, h_n)
    for s, n in enumerate(lens):
        packed = (n // r_len) * r_len
        assert O.ring_split(n, r_len) == (packed, n - packed)
        pos = np.arange(packed)
        O.store_kv(layer, k[s][:packed], v[s][:packed], table[s][pos // 16] * 16 + pos % 16, want)
        np.testing.assert_array_equal(ring_k[s, :n - packed], k[s][packed:])
        np.testing.assert_array_equal(ring_v[s, :n - packed], v[s][packed:])
    np.testing.assert_array_equal(cache.data, want.data)
    assert cache.data.any()


def test_ring_chunked_append_equals_steps():
    """A prefill chunk and a later chunk give the state that single-token
    steps give (the chunk crosses two ring blocks)."""
    cfg = O.Config(head_dim=16, key_quant_bits=8, value_quant_bits=3)
    layer = O.make_layer(cfg, 0)
    lens, r_len, h_n = [100], 32, 1
    k, v = _ring_inputs(np.random.default_rng(22), lens, h_n, 16)
    c1, table, rk1, rv1 = _ring_setup(layer, lens, h_n, r_len)
    O.ring_append(layer, c1, table, rk1, rv1, np.array([0]), k[0][:45], v[0][:45], np.array([0, 45]))
    O.ring_append(layer, c1, table, rk1, rv1, np.array([45]), k[0][45:], v[0][45:], np.array([0, 55]))
    c2, _, rk2, rv2 = _ring_setup(layer, lens, h_n, r_len)
    for p in range(100):
        O.ring_append(layer, c2, table, rk2, rv2, np.array([p]), k[0][p:p + 1], v[0][p:p + 1], np.array([0, 1]))
    np.testing.assert_array_equal(c1.data, c2.data)
    np.testing.assert_array_equal(rk1[:, :100 % r_len], rk2[:, :100 % r_len])
    np.testing.assert_array_equal(rv1[:, :100 % r_len], rv2[:, :100 % r_len])


def test_ring_decode_reduces_to_packed_decode_and_closed_forms():
    cfg = O.Config(head_dim=16, key_quant_bits=4, value_quant_bits=4, norm_correction=True)
    layer = O.make_layer(cfg, 0)
    lens, r_len, h_n = [64, 1, 20], 32, 1
    k, v = _ring_inputs(np.random.default_rng(23), lens, h_n, 16)
    k[2][:] = k[2][:1]  # identical keys in the third sequence's ring
    cache, table, ring_k, ring_v = _ring_setup(layer, lens, h_n, r_len)
    cu = np.concatenate([[0], np.cumsum(lens)])
    O.ring_append(layer, cache, table, ring_k, ring_v, np.zeros(3, dtype=np.int64), np.concatenate(k),
                  np.concatenate(v), cu)
    q = O.bf16_round(np.random.default_rng(24).standard_normal((3, 2, 16)).astype(np.float32))
    got = O.decode_attention_ring(layer, q, cache, table, np.array(lens), ring_k, ring_v)
    # 64 tokens = two whole ring blocks: nothing in the ring, the plain packed decode
    plain = O.decode_attention(layer, q, cache, table, np.array(lens))
    np.testing.assert_array_equal(got[0], plain[0])
    # one token, exact in the ring: the output is that value row
    np.testing.assert_array_equal(got[1, 0], v[1][0, 0].astype(np.float64))
    # identical exact keys: the mean of the exact values
    np.testing.assert_allclose(got[2, 1], v[2][:, 0].astype(np.float64).mean(axis=0), rtol=1e-12, atol=1e-13)
    # no tokens: zero rows
    assert not O.decode_attention_ring(layer, q, cache, table, np.array([0, 0, 0]), ring_k, ring_v).any()
