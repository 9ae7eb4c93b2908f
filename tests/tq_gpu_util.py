"""Helpers shared by the GPU parity tests: run the CUDA path through the
binding, run the oracle on the same seeded inputs, compare."""
import numpy as np
import torch

import kv_cache_quantization_store_gb300 as tq
import oracle as O

DECODE_RTOL = 2e-3  # max |o - r| / max |r| per output row


def oracle_layer(wl, layer_idx):
    cfg = O.Config(head_dim=wl.head_dim, key_quant_bits=wl.key_bits, value_quant_bits=wl.value_bits,
                   seed=wl.seed, norm_correction=wl.norm_correction)
    return O.make_layer(cfg, layer_idx)


def host_cfg(wl):
    return tq.tq_config_init(wl.head_dim, wl.key_bits, wl.value_bits, wl.norm_correction, wl.seed)


def bf16(x, device):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).to(device)


def gpu_cache_for(wl, cfg, layer_idx, device, num_blocks=None):
    _, nblk = wl.layout()
    return tq.new_paged_cache(cfg, num_blocks or nblk, wl.block_size, wl.num_kv_heads, layer_idx,
                              block_stride=wl.block_stride, device=device)


def gpu_store(wl, layer_idx, device, k, v, slots=None, cache=None):
    cfg = host_cfg(wl)
    cache = cache or gpu_cache_for(wl, cfg, layer_idx, device)
    sm = wl.slot_mapping() if slots is None else slots
    tq.tq_store_kv(cfg, bf16(k, device), bf16(v, device), torch.from_numpy(np.asarray(sm, dtype=np.int64)).to(device),
                   cache)
    torch.cuda.synchronize()
    return cfg, cache


def oracle_cache(wl, layer, k, v):
    _, nblk = wl.layout()
    cache = O.new_cache(layer.cfg, nblk, wl.block_size, wl.num_kv_heads, wl.block_stride)
    near = O.store_kv(layer, k, v, wl.slot_mapping(), cache)
    return cache, near


def slot_bytes(flat: np.ndarray, wl, slot_al: int, slots: np.ndarray) -> np.ndarray:
    """Bytes [T, H, slot_al] of every KV head's slot at the given slot ids,
    read from a flat cache copy."""
    h_n = wl.num_kv_heads
    stride = wl.block_stride or wl.block_size * h_n * slot_al
    blk, pos = np.divmod(np.asarray(slots, dtype=np.int64), wl.block_size)
    off = (blk * stride)[:, None] + (pos[:, None] * h_n + np.arange(h_n)[None, :]) * slot_al
    return flat[off[..., None] + np.arange(slot_al)]


def norm_midpoint_window(k64: np.ndarray) -> np.ndarray:
    """vec_norm exemption: the fp64 norm lies within 1e-5 relative of an
    fp16 rounding midpoint (the two ends of the window round differently)."""
    n = np.linalg.norm(k64, axis=-1)
    return np.float16(n * (1 - 1e-5)) != np.float16(n * (1 + 1e-5))


def compare_slots(layer, got: np.ndarray, want: np.ndarray, near: np.ndarray, k: np.ndarray):
    """Bit-exact slot bytes, except key indices inside the near-boundary
    window and vec_norm within one fp16 ulp next to a rounding midpoint.
    got/want: [N, slot]; near/k: [N, d].  Returns exemption counts."""
    cfg = layer.cfg
    kp = cfg.key_packed_size
    np.testing.assert_array_equal(got[:, kp:], want[:, kp:], err_msg="value bytes differ")
    if cfg.key_fp8:
        np.testing.assert_array_equal(got[:, :kp], want[:, :kp], err_msg="fp8 key bytes differ")
        return {"index_exempt": 0, "norm_exempt": 0}
    nb = kp - 2
    gi = O.unpack_bits(got[:, :nb], cfg.key_mse_bits, cfg.head_dim)
    wi = O.unpack_bits(want[:, :nb], cfg.key_mse_bits, cfg.head_dim)
    bad = (gi != wi) & ~near
    assert not bad.any(), f"{int(bad.sum())} key indices differ outside the boundary window, first at {np.argwhere(bad)[:4]}"
    gn = got[:, nb:nb + 2].copy().view("<u2").astype(np.int64).ravel()
    wn = want[:, nb:nb + 2].copy().view("<u2").astype(np.int64).ravel()
    win = norm_midpoint_window(np.asarray(k, dtype=np.float64))
    ok = (gn == wn) | ((np.abs(gn - wn) == 1) & win)
    assert ok.all(), f"{int((~ok).sum())} vec_norm values differ"
    return {"index_exempt": int((gi != wi).sum()), "norm_exempt": int((gn != wn).sum())}


def gpu_decode(wl, cfg, cache, q, device, num_splits=0, seq_lens=None, max_seq_len=None, table=None):
    table = wl.layout()[0] if table is None else table
    lens = wl.seq_lens if seq_lens is None else np.asarray(seq_lens)
    max_len = int(lens.max()) if max_seq_len is None else int(max_seq_len)
    s, hq, d = q.shape
    ws = torch.zeros(tq.tq_decode_workspace_size(cfg, s, hq, wl.num_kv_heads, wl.block_size, max_len, num_splits),
                     dtype=torch.uint8, device=device)
    out = torch.full((s, hq, d), float("nan"), dtype=torch.float32, device=device)
    tq.tq_decode_attention(cfg, bf16(q, device), cache, torch.from_numpy(table.astype(np.int32)).to(device),
                           torch.from_numpy(lens.astype(np.int32)).to(device), max_len, out, ws,
                           num_splits=num_splits)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def assert_rows_close(got: np.ndarray, want: np.ndarray, rtol=DECODE_RTOL, rows=None):
    """Per output row: max |got - want| <= rtol * max |want| (rows of zeros must be zero)."""
    got = got.reshape(-1, got.shape[-1]) if rows is None else np.stack([got[r] for r in rows])
    want = want.reshape(-1, want.shape[-1]) if rows is None else np.stack([want[r] for r in rows])
    assert np.all(np.isfinite(got)), "non-finite decode output"
    err = np.abs(got - want).max(axis=1)
    scale = np.abs(want).max(axis=1)
    rel = np.where(scale > 0, err / np.where(scale > 0, scale, 1), err)
    assert rel.max() <= rtol, f"max row error {rel.max():.3e} at row {int(rel.argmax())}"
    return float(rel.max())


def upload_cache(ocache, cfg, layer_idx, device):
    """A device copy of an oracle-written cache (the GPU decodes the oracle's bytes)."""
    c = tq.PagedCache(torch.from_numpy(ocache.data.copy()).to(device), ocache.num_blocks, ocache.block_size,
                      ocache.num_kv_heads, layer_idx, ocache.block_stride,
                      torch.zeros(1, dtype=torch.int32, device=device))
    return c
