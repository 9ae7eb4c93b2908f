"""Parity at the five configurations' full sizes, in the launch
configuration bench.py times (one store of every token, the whole decode
batch with the automatic split count), on sampled outputs.

Store: the slots of a random sample of tokens (all KV heads) against the
oracle's encoding of the same rows, with the store's exemptions.  Decode:
for a few sampled (sequence, KV head) pairs the oracle encodes the whole
history of that head and its bytes replace the GPU's in the device cache,
so the GPU decodes oracle bytes there.  The GPU then decodes the full batch,
and the rows of those query heads are compared with the oracle's decode
within the decode tolerance.  No oracle input comes from the CUDA path.
"""
import math

import numpy as np
import pytest
import torch

import kv_cache_quantization_store_gb300 as tq
import oracle as O
from kv_cache_quantization_store_gb300 import workloads as W
from tq_gpu_util import (assert_rows_close, bf16, compare_slots, gpu_decode, gpu_store, host_cfg, oracle_layer,
                         slot_bytes)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

#: configuration -> (sampled sequences, sampled KV heads per sequence, sampled store tokens)
SAMPLES = {"c1": (2, 2, 256), "c2": (1, 2, 256), "c3": (1, 1, 256), "c4": (3, 2, 256)}


@pytest.mark.parametrize("name", list(SAMPLES))
def test_full_size_store_and_decode(cuda_device, name):
    n_seq, n_head, n_tok = SAMPLES[name]
    wl = W.named(name)
    layer_idx = wl.layers[-1]
    k, v = wl.kv()
    cfg, cache = gpu_store(wl, layer_idx, cuda_device, k, v)
    assert cache.error_flags() == 0
    layer = oracle_layer(wl, layer_idx)
    h_n, d, slot_al = wl.num_kv_heads, wl.head_dim, cfg.slot_size_aligned
    rng = np.random.default_rng(5000 + int(name[1]))
    sm = wl.slot_mapping()

    # ---- store: sampled tokens, every head -----------------------------------------
    tok = np.sort(rng.choice(wl.num_tokens, n_tok, replace=False))
    want, near = O.encode_slots(layer, k[tok].reshape(-1, d), v[tok].reshape(-1, d))
    flat = cache.data.cpu().numpy()
    got = slot_bytes(flat, wl, slot_al, sm[tok]).reshape(-1, slot_al)
    compare_slots(layer, got, want, near, k[tok].reshape(-1, d))

    # ---- decode: oracle bytes for the sampled (sequence, head) histories ------------
    table, nblk = wl.layout()
    cu = wl.cu_seqlens()
    ocache = O.new_cache(layer.cfg, nblk, wl.block_size, h_n, wl.block_stride)
    seqs = rng.choice(wl.num_seqs, n_seq, replace=False)
    group = wl.num_q_heads // h_n
    rows = []
    data = cache.data
    for s in seqs:
        n = int(wl.seq_lens[s])
        pos = np.arange(n)
        ids = table[s][pos // wl.block_size].astype(np.int64) * wl.block_size + pos % wl.block_size
        for h in rng.choice(h_n, n_head, replace=False):
            slots, _ = O.encode_slots(layer, k[cu[s]:cu[s] + n, h], v[cu[s]:cu[s] + n, h])
            off = O.slot_offsets(ocache, ids)[:, h]
            idx = (off[:, None] + np.arange(slot_al)).ravel()
            ocache.data[idx] = slots.ravel()
            data[torch.from_numpy(idx).to(cuda_device)] = torch.from_numpy(slots.ravel()).to(cuda_device)
            rows += [(int(s), int(hq)) for hq in range(h * group, (h + 1) * group)]
    q = wl.q()
    got = gpu_decode(wl, cfg, cache, q, cuda_device)  # automatic split count, the whole batch
    assert np.all(np.isfinite(got))
    want = O.decode_attention(layer, q, ocache, table, wl.seq_lens, rows=rows)
    assert_rows_close(got, want, rows=rows)
    assert cache.error_flags() == 0


#: configuration -> sampled sequences (one 16-token window per grid-stride range of each)
DEQUANT_SAMPLES = {"c3": 2, "c4": 6, "c2": 2}


def _dequant_steps(wl):
    """Grid-stride ranges of the dequant's full-size launch, as positions:
    (steps per warp, positions one step of the grid covers).  Mirrors the
    staged launch in tq_dequant.cu: token steps of ts = 16 / gcd(H * slot, 16)
    positions, 8 warps per block, about 8 blocks per SM across all sequences,
    at most one step per warp per block column."""
    cfg = host_cfg(wl)
    ts = 16 // math.gcd(wl.num_kv_heads * cfg.slot_size_aligned, 16)
    steps_n = -(-int(wl.seq_lens.max()) // ts)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    gx = -(-sms * 8 // wl.num_seqs)
    gx = max(1, min(gx, -(-steps_n // 8), 65535))
    per_step = gx * 8 * ts
    steps = -(-steps_n // (gx * 8))
    return steps, per_step


@pytest.mark.parametrize("name", list(DEQUANT_SAMPLES))
def test_full_size_dequant(cuda_device, name):
    """tq_dequant over the whole decode batch in its full-size launch shape
    (several grid-stride steps per warp and the 1024-block cap at c3):
    oracle-encoded slots at sampled positions, one 16-token window in each
    grid-stride range of each sampled sequence, all KV heads, compared with
    the oracle's dequant of the same bytes (values bit-exact, keys within one
    bf16 ulp)."""
    n_seq = DEQUANT_SAMPLES[name]
    wl = W.named(name)
    layer_idx = wl.layers[0]
    layer = oracle_layer(wl, layer_idx)
    cfg = host_cfg(wl)
    h_n, d, slot_al = wl.num_kv_heads, wl.head_dim, cfg.slot_size_aligned
    table, nblk = wl.layout()
    cu = wl.cu_seqlens()
    steps, per_step = _dequant_steps(wl)
    if name in ("c3", "c4"):
        assert steps >= 4, (name, steps)  # the multi-step path is the one under test
    rng = np.random.default_rng(7000 + int(name[1]))
    seqs = np.sort(rng.choice(wl.num_seqs, n_seq, replace=False))
    ocache = O.new_cache(layer.cfg, nblk, wl.block_size, h_n, wl.block_stride)
    picked = []  # (sequence, positions)
    for s in seqs:
        n = int(wl.seq_lens[s])
        pos = []
        for i in range(steps):
            lo, hi = i * per_step, min(n, (i + 1) * per_step)
            if hi - lo >= 16:
                p0 = lo + 16 * int(rng.integers(0, (hi - lo) // 16))
                pos.extend(range(p0, p0 + 16))
        pos = np.array(pos, dtype=np.int64)
        picked.append((int(s), pos))
        k = np.concatenate([wl.kv(int(cu[s] + p), int(cu[s] + p + 16))[0] for p in pos[::16]])
        v = np.concatenate([wl.kv(int(cu[s] + p), int(cu[s] + p + 16))[1] for p in pos[::16]])
        ids = table[s][pos // wl.block_size].astype(np.int64) * wl.block_size + pos % wl.block_size
        off = O.slot_offsets(ocache, ids)
        for h in range(h_n):
            slots, _ = O.encode_slots(layer, k[:, h], v[:, h])
            ocache.data[(off[:, h][:, None] + np.arange(slot_al)).ravel()] = slots.ravel()
    cache = tq.new_paged_cache(cfg, nblk, wl.block_size, h_n, layer_idx, block_stride=wl.block_stride,
                               device=cuda_device)
    cache.data.copy_(torch.from_numpy(ocache.data))
    rows = int(cu[-1])
    k_out = torch.full((rows, h_n, d), float("nan"), dtype=torch.bfloat16, device=cuda_device)
    v_out = torch.full_like(k_out, float("nan"))
    tq.tq_dequant(cfg, cache, torch.from_numpy(table).to(cuda_device), torch.from_numpy(cu).to(cuda_device),
                  int(wl.seq_lens.max()), k_out, v_out)
    torch.cuda.synchronize()
    assert cache.error_flags() == 0
    for s, pos in picked:
        r = torch.from_numpy(cu[s] + pos).to(cuda_device)
        kg = k_out[r].float().cpu().numpy()
        vg = v_out[r].float().cpu().numpy()
        for h in range(h_n):
            sl = O.read_slots(ocache, table[s], int(pos[-1]) + 1, h)[pos]
            k_hat, _ = O.dequant_slots(layer, sl)
            kw = O.bf16_round(k_hat.astype(np.float32))
            vw = O.bf16_round(O.dequant_values_f32(layer, sl))
            np.testing.assert_array_equal(vg[:, h], vw, err_msg=f"values, sequence {s} head {h}")
            tol = np.abs(kw) * 2.0 ** -7 + 1e-6 * np.abs(kw).max(axis=-1, keepdims=True)
            assert np.all(np.abs(kg[:, h] - kw) <= tol), f"keys, sequence {s} head {h}"
