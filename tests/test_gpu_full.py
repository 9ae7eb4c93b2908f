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
