"""The dequant-then-dense comparison path ([ART] hnwysp.cn TurboQuant
article, "Obstacle 1": the whole history expanded to full precision before
ordinary attention) against the CPU oracle.

- The dense kernel alone: the oracle's own bf16 rows (O.dequant_cache) are
  uploaded as its K and V, and its output is compared with brute-force fp64
  attention over those same rows; only the kernel's fp32 arithmetic
  differs, so rows agree to 1e-5 of their largest entry.
- The whole path (tq_dequant on the oracle's packed cache, then the dense
  kernel) against the oracle's decode of the packed cache
  (O.decode_attention).  The dequant rounds values to bf16 (relative error
  at most u = 2^-9) and keys to within one bf16 ulp of the oracle's bf16
  rounding (at most 3u from the exact key).  A key error moves each logit by
  at most D = 3u * sm_scale * max_t sum_i |q_i k_ti| and softmax weights by a
  factor within exp(+-2D), so per output row
      |o - r| <= (exp(2D) - 1) max_t |v_t| + u max_t |v_t|,
  checked on top of the fused decode's 2e-3 of max |r|.  The fused decode
  reads the packed bytes and has no such term.
"""
import numpy as np
import pytest
import torch

import kv_cache_quantization_store_gb300 as tq
import oracle as O
from kv_cache_quantization_store_gb300 import workloads as W
from tq_gpu_util import assert_rows_close, bf16, host_cfg, oracle_cache, oracle_layer, upload_cache

pytestmark = pytest.mark.gpu

CASES = [
    W.named("c0"),
    W.small("c1", [1, 15, 16, 17, 250, 700]),
    W.small("c2", [33, 513, 2]),
    W.small("c3", [1000, 77, 0]),
    W.small("c4", [600, 31], layers=(2,)),
    W.custom(16, 3, 3, False, 2, 2, 16, [40, 3], 2001),
    W.custom(32, 4, 3, True, 1, 8, 32, [100], 2002),
    W.custom(64, 4, 3, True, 4, 20, 16, [65, 130, 5], 2003),
]
IDS = [f"{w.name}-{'x'.join(map(str, w.seq_lens))}" for w in CASES]


def _dense_from_rows(wl, q, k_rows, v_rows, cu, dev):
    max_len = max(1, int(wl.seq_lens.max()))
    ws = torch.zeros(tq.tq_dense_decode_workspace_size(wl.head_dim, wl.num_seqs, wl.num_q_heads,
                                                       wl.num_kv_heads, max_len), dtype=torch.uint8, device=dev)
    out = torch.full((wl.num_seqs, wl.num_q_heads, wl.head_dim), float("nan"), dtype=torch.float32, device=dev)
    tq.tq_dense_decode_attention(bf16(q, dev), k_rows, v_rows, torch.from_numpy(cu).to(dev), max_len, out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _setup(wl, dev):
    layer_idx = wl.layers[-1]
    k, v = wl.kv()
    layer = oracle_layer(wl, layer_idx)
    ocache, _ = oracle_cache(wl, layer, k, v)
    return layer, ocache, wl.q(), wl.layout()[0], wl.cu_seqlens()


@pytest.mark.parametrize("wl", CASES, ids=IDS)
def test_dense_kernel_on_oracle_rows(cuda_device, wl):
    layer, ocache, q, table, cu = _setup(wl, cuda_device)
    kd, vd = O.dequant_cache(layer, ocache, table, cu)
    rows = max(1, int(cu[-1]))
    k_rows = torch.zeros((rows, wl.num_kv_heads, wl.head_dim), dtype=torch.bfloat16, device=cuda_device)
    v_rows = torch.zeros_like(k_rows)
    if cu[-1] > 0:
        k_rows[: int(cu[-1])] = bf16(kd, cuda_device)
        v_rows[: int(cu[-1])] = bf16(vd, cuda_device)
    got = _dense_from_rows(wl, q, k_rows, v_rows, cu, cuda_device)
    g = wl.num_q_heads // wl.num_kv_heads
    sm = 1.0 / np.sqrt(wl.head_dim)
    exact = np.zeros_like(got, dtype=np.float64)
    for s in range(wl.num_seqs):
        a, b = int(cu[s]), int(cu[s + 1])
        for hq in range(wl.num_q_heads):
            exact[s, hq] = O.attention_row(q[s, hq], kd[a:b, hq // g].astype(np.float64),
                                           vd[a:b, hq // g].astype(np.float64), sm)
    assert_rows_close(got, exact, rtol=1e-5)


@pytest.mark.parametrize("wl", CASES, ids=IDS)
def test_dequant_then_dense_against_oracle_decode(cuda_device, wl):
    layer, ocache, q, table, cu = _setup(wl, cuda_device)
    cfg = host_cfg(wl)
    cache = upload_cache(ocache, cfg, wl.layers[-1], cuda_device)
    rows = max(1, int(cu[-1]))
    max_len = max(1, int(wl.seq_lens.max()))
    k_rows = torch.empty((rows, wl.num_kv_heads, wl.head_dim), dtype=torch.bfloat16, device=cuda_device)
    v_rows = torch.empty_like(k_rows)
    tq.tq_dequant(cfg, cache, torch.from_numpy(table).to(cuda_device), torch.from_numpy(cu).to(cuda_device), max_len,
                  k_rows, v_rows)
    got = _dense_from_rows(wl, q, k_rows, v_rows, cu, cuda_device)
    assert cache.error_flags() == 0
    assert np.all(np.isfinite(got))
    want = O.decode_attention(layer, q, ocache, table, wl.seq_lens)
    g = wl.num_q_heads // wl.num_kv_heads
    sm = 1.0 / np.sqrt(wl.head_dim)
    u = 2.0 ** -9
    for s in range(wl.num_seqs):
        a, b = int(cu[s]), int(cu[s + 1])
        for hq in range(wl.num_q_heads):
            if b == a:
                assert not got[s, hq].any()
                continue
            k_hat, v_hat = O.dequant_slots(layer, O.read_slots(ocache, table[s], b - a, hq // g))
            logit_shift = 3 * u * sm * np.max(np.abs(k_hat) @ np.abs(q[s, hq].astype(np.float64)))
            bound = (np.expm1(2 * logit_shift) + u) * np.abs(v_hat).max() + 2e-3 * np.abs(want[s, hq]).max()
            assert np.abs(got[s, hq] - want[s, hq]).max() <= bound, (s, hq)
