"""CUDA path against the CPU oracle on the same seeded inputs.

Store: packed bytes bit-exact (values, FP8 keys), key indices bit-exact
outside the near-boundary window, vec_norm bit-exact outside the fp16
midpoint window.  Decode: per output row max |o - r| <= 2e-3 max |r|,
where the GPU decodes the oracle's own cache bytes (small cases) or its own
cache (full sizes, sampled rows).  Dequant: values bit-exact in bf16, keys
within one bf16 ulp.
"""
import math

import numpy as np
import pytest
import torch

import kv_cache_quantization_store_gb300 as tq
import oracle as O
from kv_cache_quantization_store_gb300 import workloads as W
from tq_gpu_util import (assert_rows_close, bf16, compare_slots, gpu_cache_for, gpu_decode, gpu_store, host_cfg,
                         oracle_cache, oracle_layer, slot_bytes, upload_cache)

pytestmark = pytest.mark.gpu


def small_cases():
    return [
        W.named("c0"),
        W.small("c1", [1, 15, 16, 17, 250, 700]),
        W.small("c2", [33, 513, 2]),
        W.small("c3", [1000, 77]),
        W.small("c4", [600, 31], layers=(2,)),
        W.custom(16, 3, 3, False, 2, 2, 16, [40, 3], 2001),
        W.custom(32, 4, 3, True, 1, 8, 32, [100], 2002),
        W.custom(64, 4, 3, True, 4, 20, 16, [65, 130, 5], 2003),
        W.custom(128, 8, 3, False, 3, 6, 16, [90, 47], 2004, kv_mode="lognormal"),
        W.custom(256, 8, 4, False, 2, 16, 48, [200], 2005),
        W.custom(256, 3, 3, True, 1, 1, 16, [77], 2006, kv_mode="outliers"),
        W.custom(128, 4, 4, False, 8, 64, 64, [300, 129], 2007),
        # 4-bit keys in the paired-word decode: every warp's key share
        # 2 bytes off a word (H = 1), and even / odd heads mixed (H = 2, 4)
        W.custom(256, 4, 4, True, 1, 4, 16, [300, 17], 2011),
        W.custom(256, 4, 4, True, 2, 4, 32, [129, 64], 2012),
        W.custom(128, 4, 4, True, 4, 16, 16, [97, 250], 2013),
    ]


CASES = small_cases()
IDS = [f"{w.name}-{'x'.join(map(str, w.seq_lens))}" for w in CASES]


@pytest.mark.parametrize("wl", CASES, ids=IDS)
def test_store_parity(cuda_device, wl):
    layer_idx = wl.layers[-1]
    k, v = wl.kv()
    cfg, cache = gpu_store(wl, layer_idx, cuda_device, k, v)
    layer = oracle_layer(wl, layer_idx)
    ocache, near = oracle_cache(wl, layer, k, v)
    assert cache.error_flags() == 0
    flat = cache.data.cpu().numpy()
    sm = wl.slot_mapping()
    got = slot_bytes(flat, wl, cfg.slot_size_aligned, sm).reshape(-1, cfg.slot_size_aligned)
    want = slot_bytes(ocache.data, wl, cfg.slot_size_aligned, sm).reshape(-1, cfg.slot_size_aligned)
    stats = compare_slots(layer, got, want, near.reshape(-1, wl.head_dim), k.reshape(-1, wl.head_dim))
    assert stats["index_exempt"] <= max(2, got.shape[0] * wl.head_dim // 100000)
    # bytes outside written slots stay zero
    written = np.zeros(flat.shape, dtype=bool)
    idx = slot_bytes(np.arange(flat.size), wl, cfg.slot_size_aligned, sm)
    written[idx.ravel()] = True
    assert not flat[~written].any()


@pytest.mark.parametrize("wl", CASES, ids=IDS)
def test_decode_parity(cuda_device, wl):
    layer_idx = wl.layers[-1]
    k, v = wl.kv()
    layer = oracle_layer(wl, layer_idx)
    ocache, _ = oracle_cache(wl, layer, k, v)
    cfg = host_cfg(wl)
    cache = upload_cache(ocache, cfg, layer_idx, cuda_device)
    q = wl.q()
    table = wl.layout()[0]
    want = O.decode_attention(layer, q, ocache, table, wl.seq_lens)
    for splits in (0, 1, 3):
        got = gpu_decode(wl, cfg, cache, q, cuda_device, num_splits=splits)
        assert_rows_close(got, want)
    assert cache.error_flags() == 0


@pytest.mark.parametrize("wl", CASES[:6], ids=IDS[:6])
def test_decode_any_split_count(cuda_device, wl):
    """Every split count, up to one split per 16-token chunk, matches the
    oracle (the partial states merge by log-sum-exp)."""
    layer_idx = wl.layers[-1]
    k, v = wl.kv()
    layer = oracle_layer(wl, layer_idx)
    ocache, _ = oracle_cache(wl, layer, k, v)
    cfg = host_cfg(wl)
    cache = upload_cache(ocache, cfg, layer_idx, cuda_device)
    q = wl.q()
    want = O.decode_attention(layer, q, ocache, wl.layout()[0], wl.seq_lens)
    max_chunks = math.ceil(int(wl.seq_lens.max()) / 16)
    for splits in sorted({2, 7, max_chunks}):
        assert_rows_close(gpu_decode(wl, cfg, cache, q, cuda_device, num_splits=splits), want)


@pytest.mark.parametrize("splits", [300, 520])
def test_decode_more_splits_than_combine_lanes(cuda_device, splits):
    """More splits than the combine's 8 warps x 32 lanes: each lane folds
    several splits' (m, l); the short sequences leave most splits empty."""
    wl = W.custom(64, 4, 4, True, 2, 8, 16, [8300, 40, 1], 2008)
    layer_idx = wl.layers[-1]
    k, v = wl.kv()
    layer = oracle_layer(wl, layer_idx)
    ocache, _ = oracle_cache(wl, layer, k, v)
    cfg = host_cfg(wl)
    cache = upload_cache(ocache, cfg, layer_idx, cuda_device)
    q = wl.q()
    want = O.decode_attention(layer, q, ocache, wl.layout()[0], wl.seq_lens)
    assert_rows_close(gpu_decode(wl, cfg, cache, q, cuda_device, num_splits=splits), want)
    assert cache.error_flags() == 0


@pytest.mark.parametrize("wl", CASES, ids=IDS)
def test_dequant_parity(cuda_device, wl):
    layer_idx = wl.layers[-1]
    k, v = wl.kv()
    layer = oracle_layer(wl, layer_idx)
    ocache, _ = oracle_cache(wl, layer, k, v)
    cfg = host_cfg(wl)
    cache = upload_cache(ocache, cfg, layer_idx, cuda_device)
    table = wl.layout()[0]
    cu = wl.cu_seqlens()
    rows = int(cu[-1])
    k_out = torch.full((rows, wl.num_kv_heads, wl.head_dim), float("nan"), dtype=torch.bfloat16, device=cuda_device)
    v_out = torch.full_like(k_out, float("nan"))
    tq.tq_dequant(cfg, cache, torch.from_numpy(table).to(cuda_device), torch.from_numpy(cu).to(cuda_device),
                  int(wl.seq_lens.max()), k_out, v_out)
    torch.cuda.synchronize()
    kw, vw = O.dequant_cache(layer, ocache, table, cu)
    kg = k_out.float().cpu().numpy()
    vg = v_out.float().cpu().numpy()
    np.testing.assert_array_equal(vg, vw)
    tol = np.abs(kw) * 2.0 ** -7 + 1e-6 * np.abs(kw).max(axis=-1, keepdims=True)
    assert np.all(np.abs(kg - kw) <= tol)


@pytest.mark.parametrize("wl", [c for c in CASES if c.head_dim >= 64], ids=[i for c, i in zip(CASES, IDS)
                                                                      if c.head_dim >= 64])
def test_dequant_parity_16_byte_aligned_outputs(cuda_device, wl):
    """Outputs that start 16 bytes past a 32-byte boundary (the least
    alignment tq_dequant accepts): every 16-byte group store lands in place
    and nothing is written before the first row."""
    layer_idx = wl.layers[-1]
    k, v = wl.kv()
    layer = oracle_layer(wl, layer_idx)
    ocache, _ = oracle_cache(wl, layer, k, v)
    cfg = host_cfg(wl)
    cache = upload_cache(ocache, cfg, layer_idx, cuda_device)
    table = wl.layout()[0]
    cu = wl.cu_seqlens()
    rows = int(cu[-1])
    n = rows * wl.num_kv_heads * wl.head_dim
    kbuf = torch.full((n + 8,), float("nan"), dtype=torch.bfloat16, device=cuda_device)
    vbuf = torch.full_like(kbuf, float("nan"))
    assert kbuf.data_ptr() % 32 == 0
    k_out = kbuf[8:].view(rows, wl.num_kv_heads, wl.head_dim)  # 16 bytes past the boundary
    v_out = vbuf[8:].view(rows, wl.num_kv_heads, wl.head_dim)
    tq.tq_dequant(cfg, cache, torch.from_numpy(table).to(cuda_device), torch.from_numpy(cu).to(cuda_device),
                  int(wl.seq_lens.max()), k_out, v_out)
    torch.cuda.synchronize()
    kw, vw = O.dequant_cache(layer, ocache, table, cu)
    np.testing.assert_array_equal(v_out.float().cpu().numpy(), vw)
    kg = k_out.float().cpu().numpy()
    tol = np.abs(kw) * 2.0 ** -7 + 1e-6 * np.abs(kw).max(axis=-1, keepdims=True)
    assert np.all(np.abs(kg - kw) <= tol)
    assert torch.isnan(kbuf[:8].float()).all() and torch.isnan(vbuf[:8].float()).all()  # nothing before the rows


def test_fp8_keys_exhaustive_bf16(cuda_device):
    """All finite bf16 bit patterns as FP8 keys (d=128, 512 vectors)."""
    pat = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        x = (pat << 16).view(np.float32)
    x = np.where(np.isfinite(x) | np.isinf(x), x, 0).astype(np.float32)
    wl = W.custom(128, 8, 4, False, 1, 1, 16, [512], 2100)
    k = x.reshape(512, 1, 128)
    _, v = wl.kv()
    cfg, cache = gpu_store(wl, 0, cuda_device, k, v)
    got = slot_bytes(cache.data.cpu().numpy(), wl, cfg.slot_size_aligned, wl.slot_mapping()).reshape(512, -1)
    want = O.e4m3_encode(k.reshape(-1)).reshape(512, 128)
    np.testing.assert_array_equal(got[:, :128], want)


def test_negative_and_out_of_range_slots(cuda_device):
    wl = W.custom(64, 3, 4, False, 2, 4, 16, [64], 2200)
    k, v = wl.kv()
    sm = wl.slot_mapping().copy()
    sm[5] = -1
    sm[9] = 10 ** 9  # beyond the cache: skipped and flagged
    cfg, cache = gpu_store(wl, 0, cuda_device, k, v, slots=sm)
    assert cache.error_flags() & tq.TQ_FLAG_SLOT_OUT_OF_RANGE
    layer = oracle_layer(wl, 0)
    keep = np.ones(64, dtype=bool)
    keep[[5, 9]] = False
    ocache = O.new_cache(layer.cfg, wl.layout()[1], wl.block_size, wl.num_kv_heads)
    near = O.store_kv(layer, k, v, np.where(keep, sm, -1), ocache)
    flat = cache.data.cpu().numpy()
    orig = wl.slot_mapping()
    assert not slot_bytes(flat, wl, cfg.slot_size_aligned, orig[~keep]).any()
    got = slot_bytes(flat, wl, cfg.slot_size_aligned, orig[keep]).reshape(-1, cfg.slot_size_aligned)
    want = slot_bytes(ocache.data, wl, cfg.slot_size_aligned, orig[keep]).reshape(-1, cfg.slot_size_aligned)
    compare_slots(layer, got, want, near[keep].reshape(-1, 64), k[keep].reshape(-1, 64))


def test_decode_flags_bad_block_and_length(cuda_device):
    wl = W.custom(64, 3, 4, False, 1, 2, 16, [48, 20], 2300)
    k, v = wl.kv()
    cfg, cache = gpu_store(wl, 0, cuda_device, k, v)
    table = wl.layout()[0].copy()
    table[0, 1] = 10 ** 6
    out = gpu_decode(wl, cfg, cache, wl.q(), cuda_device, table=table)
    assert np.all(np.isfinite(out))
    assert cache.error_flags() & tq.TQ_FLAG_BLOCK_OUT_OF_RANGE
    cache.flags.zero_()
    out = gpu_decode(wl, cfg, cache, wl.q(), cuda_device, seq_lens=[48, 20], max_seq_len=32)
    assert np.all(np.isfinite(out))
    assert cache.error_flags() & tq.TQ_FLAG_SEQ_TOO_LONG


def test_padded_block_stride(cuda_device):
    """The lcm page geometry read the other way: 16-token blocks padded to
    the 536576-byte unified page (4bit_nc, d=256, 4 KV heads)."""
    base = W.named("c4")
    cfg = host_cfg(base)
    page, _ = tq.tq_hybrid_page(cfg, 4, 2)
    wl = W.custom(256, 4, 4, True, 4, 16, 16, [70, 33], 2400, block_stride=page)
    k, v = wl.kv()
    cfg, cache = gpu_store(wl, 1, cuda_device, k, v)
    layer = oracle_layer(wl, 1)
    ocache, near = oracle_cache(wl, layer, k, v)
    flat = cache.data.cpu().numpy()
    sm = wl.slot_mapping()
    got = slot_bytes(flat, wl, cfg.slot_size_aligned, sm).reshape(-1, cfg.slot_size_aligned)
    want = slot_bytes(ocache.data, wl, cfg.slot_size_aligned, sm).reshape(-1, cfg.slot_size_aligned)
    compare_slots(layer, got, want, near.reshape(-1, 256), k.reshape(-1, 256))
    q = wl.q()
    want_out = O.decode_attention(layer, q, ocache, wl.layout()[0], wl.seq_lens)
    dev = upload_cache(ocache, cfg, 1, cuda_device)
    assert_rows_close(gpu_decode(wl, cfg, dev, q, cuda_device), want_out)


def test_empty_inputs(cuda_device):
    wl = W.custom(64, 3, 4, False, 1, 2, 16, [16], 2500)
    cfg = host_cfg(wl)
    cache = gpu_cache_for(wl, cfg, 0, cuda_device)
    empty = torch.empty((0, 1, 64), dtype=torch.bfloat16, device=cuda_device)
    tq.tq_store_kv(cfg, empty, empty, torch.empty(0, dtype=torch.int64, device=cuda_device), cache)
    torch.cuda.synchronize()
    assert not cache.data.any()
    out = gpu_decode(wl, cfg, cache, wl.q(), cuda_device, seq_lens=[0])
    assert np.all(out == 0)


def _bf16_round(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def _bf16_step(x, steps):
    """x (bf16-representable) moved by `steps` bf16 ulps away from zero; values
    within 2 ulps of zero stay put (no step across zero into NaN patterns)."""
    b = torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    steps = np.where((b.astype(np.int32) & 0x7FFF) > 2, np.asarray(steps, dtype=np.int32), 0)
    b = (b.astype(np.int32) + steps).astype(np.int16)
    return torch.from_numpy(b).view(torch.bfloat16).float().numpy()


@pytest.mark.parametrize("vb", [3, 4])
def test_value_codes_at_quotient_ties(cuda_device, vb):
    """Value codes where (v - zero) / scale sits at, or a few bf16 steps from,
    a rounding tie k + 1/2, over thousands of scales; plus a zero scale, a
    zero point past the fp16 range and a scale past it.  Value bytes must
    equal the oracle's (IEEE fp32 division, rint half to even)."""
    d, n_tok = 64, 4096
    top = (1 << vb) - 1
    wl = W.custom(d, 3, vb, False, 1, 1, 16, [n_tok], 2600 + vb)
    rng = np.random.default_rng(2610 + vb)
    k, _ = wl.kv()
    v = np.empty((n_tok, 1, d), dtype=np.float32)
    lo = _bf16_round(-rng.uniform(0.05, 8, n_tok) * 10.0 ** rng.uniform(-3, 3, n_tok))
    hi = _bf16_round(lo + np.abs(lo) * rng.uniform(0.02, 4, n_tok))
    s = ((hi - lo).astype(np.float32) / np.float32(top)).astype(np.float16).astype(np.float32)
    z = lo.astype(np.float16).astype(np.float32)
    kk = rng.integers(0, top, (n_tok, d - 2)) + 0.5
    target = _bf16_round(z[:, None] + s[:, None] * kk)
    v[:, 0, 0], v[:, 0, 1] = lo, hi
    v[:, 0, 2:] = _bf16_step(target, rng.integers(-2, 3, target.shape))
    v[:, 0, 2:] = np.clip(v[:, 0, 2:], lo[:, None], hi[:, None])
    v[0, 0, :] = 1.25                                  # zero scale
    v[1, 0, :] = _bf16_round(rng.uniform(-2, 2, d))
    v[1, 0, 0] = -70000.0                              # zero point beyond fp16: IEEE path
    v[2, 0, :] = _bf16_round(rng.uniform(-1e4, 2e6, d))
    v[2, 0, 0], v[2, 0, 1] = -1.0e4, 2.0e6             # scale beyond fp16
    v = _bf16_round(v)
    assert np.all(np.isfinite(v))
    cfg, cache = gpu_store(wl, 0, cuda_device, k, v)
    layer = oracle_layer(wl, 0)
    ocache, near = oracle_cache(wl, layer, k, v)
    sm = wl.slot_mapping()
    got = slot_bytes(cache.data.cpu().numpy(), wl, cfg.slot_size_aligned, sm).reshape(-1, cfg.slot_size_aligned)
    want = slot_bytes(ocache.data, wl, cfg.slot_size_aligned, sm).reshape(-1, cfg.slot_size_aligned)
    compare_slots(layer, got, want, near.reshape(-1, d), k.reshape(-1, d))


@pytest.mark.parametrize("bits,lloyd_max_mse", [(3, 0.03454), (4, 0.009497)])
def test_key_distortion_matches_lloyd_max(cuda_device, bits, lloyd_max_mse):
    """Full-size property of the store + dequant path: for N(0,1) keys the
    relative key error E|k - k^|^2 / E|k|^2 is the Lloyd-Max MSE of N(0,1) at
    that width (Max 1960: 0.03454 at 8 levels, 0.009497 at 16) plus the fp16
    norm and bf16 output rounding, i.e. within a few percent."""
    from kv_cache_quantization_store_gb300 import quality
    row = quality.measure(bits, 4, 128, "normal", 16384, cuda_device, nc_options=(False,))[0]
    assert row["key_rel_mse"] == pytest.approx(lloyd_max_mse, rel=0.05)
    assert row["value_cos"] > 0.99


def test_decode_in_cuda_graph(cuda_device):
    """The decode captured in a CUDA graph (its merge kernel is launched with
    programmatic stream serialisation) replays to the eager result."""
    wl = W.small("c4", [600, 31], layers=(2,))
    layer_idx = wl.layers[-1]
    k, v = wl.kv()
    layer = oracle_layer(wl, layer_idx)
    ocache, _ = oracle_cache(wl, layer, k, v)
    cfg = host_cfg(wl)
    cache = upload_cache(ocache, cfg, layer_idx, cuda_device)
    q = bf16(wl.q(), cuda_device)
    table = torch.from_numpy(wl.layout()[0]).to(cuda_device)
    lens = torch.from_numpy(wl.seq_lens.astype(np.int32)).to(cuda_device)
    max_len = int(wl.seq_lens.max())
    for splits in (1, 4):
        ws = torch.zeros(tq.tq_decode_workspace_size(cfg, 2, wl.num_q_heads, wl.num_kv_heads, wl.block_size, max_len,
                                                     splits), dtype=torch.uint8, device=cuda_device)
        eager = torch.empty((2, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device=cuda_device)
        tq.tq_decode_attention(cfg, q, cache, table, lens, max_len, eager, ws, num_splits=splits)
        graphed = torch.full_like(eager, float("nan"))
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            tq.tq_decode_attention(cfg, q, cache, table, lens, max_len, graphed, ws, num_splits=splits)
        g.replay()
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(graphed.cpu().numpy(), eager.cpu().numpy())
    assert cache.error_flags() == 0


def test_decode_on_a_workspace_left_by_another_plan(cuda_device):
    """One workspace, never zero-filled, serves decodes with different split
    counts and batches in a row (each call writes every partial state it
    reads); the results match decodes on fresh workspaces."""
    wl = W.small("c4", [600, 31, 200], layers=(2,))
    layer_idx = wl.layers[-1]
    k, v = wl.kv()
    layer = oracle_layer(wl, layer_idx)
    ocache, _ = oracle_cache(wl, layer, k, v)
    cfg = host_cfg(wl)
    cache = upload_cache(ocache, cfg, layer_idx, cuda_device)
    q = bf16(wl.q(), cuda_device)
    table = torch.from_numpy(wl.layout()[0]).to(cuda_device)
    lens = torch.from_numpy(wl.seq_lens.astype(np.int32)).to(cuda_device)
    max_len = int(wl.seq_lens.max())
    size = max(tq.tq_decode_workspace_size(cfg, 3, wl.num_q_heads, wl.num_kv_heads, wl.block_size, max_len, sp)
               for sp in (1, 2, 5, 9))
    shared = torch.full((size,), 0x5A, dtype=torch.uint8, device=cuda_device)  # not zero-filled
    for n_seq, splits in ((3, 9), (3, 2), (1, 5), (3, 1), (2, 5)):
        fresh = torch.zeros(size, dtype=torch.uint8, device=cuda_device)
        want = torch.empty((n_seq, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device=cuda_device)
        got = torch.full_like(want, float("nan"))
        tq.tq_decode_attention(cfg, q[:n_seq], cache, table[:n_seq], lens[:n_seq], max_len, want, fresh,
                               num_splits=splits)
        tq.tq_decode_attention(cfg, q[:n_seq], cache, table[:n_seq], lens[:n_seq], max_len, got, shared,
                               num_splits=splits)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(got.cpu().numpy(), want.cpu().numpy())
    assert cache.error_flags() == 0
