"""A sweep over the kernel instantiations: every head size with a tensor-core
decode (64, 128, 256) times every (key bits, value bits) pair, each with
three different (KV heads, query group) shapes, plus CUDA-core decode shapes.  Each
case checks the store bytes, the decode (automatic split count) and the
dequant against the CPU oracle on a small ragged batch, under the same
tolerances as test_gpu_parity.py.
"""
import itertools

import numpy as np
import pytest
import torch

import kv_cache_quantization_store_gb300 as tq
import oracle as O
from kv_cache_quantization_store_gb300 import workloads as W
from tq_gpu_util import (assert_rows_close, compare_slots, gpu_decode, gpu_store, host_cfg, oracle_cache,
                         oracle_layer, slot_bytes, upload_cache)

pytestmark = pytest.mark.gpu

#: (KV heads, query heads per KV head) shapes, cycled over the cases
_HG = [(1, 4), (2, 5), (4, 1), (4, 4), (8, 2), (8, 5), (2, 8), (1, 1), (4, 8)]


def sweep_cases():
    cases = []
    pairs = [(3, 3), (3, 4), (4, 3), (4, 4), (8, 3), (8, 4)]
    for i, (d, (kb, vb), o) in enumerate(itertools.product((64, 128, 256), pairs, range(3))):
        h, g = _HG[(i // 3 + 3 * o) % len(_HG)]  # three different shapes per (d, bits)
        nc = kb != 8 and i % 2 != 0
        block = (16, 32, 64)[i % 3]
        lens = [1 + (37 * i + 11) % 211, 16 * (1 + i % 5) + i % 3]
        mode = ("normal", "outliers", "lognormal")[i % 3]
        cases.append(W.custom(d, kb, vb, nc, h, h * g, block, lens, 3000 + i, kv_mode=mode))
    # CUDA-core decode shapes (3 KV heads, or head sizes below 64)
    cases.append(W.custom(32, 4, 4, True, 3, 6, 16, [70, 5], 3100))
    cases.append(W.custom(16, 3, 4, False, 2, 6, 16, [33, 64], 3101))
    cases.append(W.custom(128, 3, 3, True, 3, 3, 32, [150, 1], 3102, kv_mode="outliers"))
    return cases


CASES = sweep_cases()
IDS = [f"{w.name}-h{w.num_kv_heads}g{w.group}-b{w.block_size}-{'x'.join(map(str, w.seq_lens))}" for w in CASES]


@pytest.mark.parametrize("wl", CASES, ids=IDS)
def test_sweep_store_decode_dequant(cuda_device, wl):
    layer_idx = wl.layers[-1]
    k, v = wl.kv()
    layer = oracle_layer(wl, layer_idx)
    ocache, near = oracle_cache(wl, layer, k, v)

    # store: packed bytes against the oracle's
    cfg, cache = gpu_store(wl, layer_idx, cuda_device, k, v)
    assert cache.error_flags() == 0
    sm = wl.slot_mapping()
    got = slot_bytes(cache.data.cpu().numpy(), wl, cfg.slot_size_aligned, sm).reshape(-1, cfg.slot_size_aligned)
    want = slot_bytes(ocache.data, wl, cfg.slot_size_aligned, sm).reshape(-1, cfg.slot_size_aligned)
    stats = compare_slots(layer, got, want, near.reshape(-1, wl.head_dim), k.reshape(-1, wl.head_dim))
    assert stats["index_exempt"] <= max(2, got.shape[0] * wl.head_dim // 100000)

    # decode of the oracle's own bytes, automatic split count
    cfg = host_cfg(wl)
    ocache_gpu = upload_cache(ocache, cfg, layer_idx, cuda_device)
    q = wl.q()
    table = wl.layout()[0]
    want_o = O.decode_attention(layer, q, ocache, table, wl.seq_lens)
    assert_rows_close(gpu_decode(wl, cfg, ocache_gpu, q, cuda_device), want_o)
    assert ocache_gpu.error_flags() == 0

    # dequant of the same bytes: values bit-exact, keys within one bf16 ulp
    cu = wl.cu_seqlens()
    rows = int(cu[-1])
    k_out = torch.full((rows, wl.num_kv_heads, wl.head_dim), float("nan"), dtype=torch.bfloat16, device=cuda_device)
    v_out = torch.full_like(k_out, float("nan"))
    tq.tq_dequant(cfg, ocache_gpu, torch.from_numpy(table).to(cuda_device), torch.from_numpy(cu).to(cuda_device),
                  int(wl.seq_lens.max()), k_out, v_out)
    torch.cuda.synchronize()
    kw, vw = O.dequant_cache(layer, ocache, table, cu)
    np.testing.assert_array_equal(v_out.float().cpu().numpy(), vw)
    kg = k_out.float().cpu().numpy()
    tol = np.abs(kw) * 2.0 ** -7 + 1e-6 * np.abs(kw).max(axis=-1, keepdims=True)
    assert np.all(np.abs(kg - kw) <= tol)
