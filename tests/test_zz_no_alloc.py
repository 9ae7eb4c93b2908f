"""The decode entry point that allocates nothing (tq_decode_attention_noalloc).

Some callers cannot give the decode a workspace: a serving engine that
handed almost all free device memory to its KV-cache pool at start-up (a
later cudaMalloc fails), a plugin inside an application that owns every
device allocation, or real-time code that cannot afford cudaMalloc's
device-wide synchronisation.  For them the library decodes on a fixed static
scratch array.  These tests call that entry point through the C ABI and
check it against the regular entry point with a caller workspace, on two
calls in a row (the scratch keeps the previous call's contents), and check
that a decode too large for the scratch is refused.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import kv_cache_quantization_store_gb300 as tq
from kv_cache_quantization_store_gb300 import workloads as W
from tq_gpu_util import DECODE_RTOL, assert_rows_close, bf16, gpu_decode, gpu_store

pytestmark = pytest.mark.gpu


def _noalloc_call(cfg, q, cache, table, lens, max_len, out, num_splits=0):
    """The C-ABI call itself: raw device pointers, the current stream."""
    desc = cache.descriptor()
    return tq.lib().tq_decode_attention_noalloc(
        ctypes.byref(cfg), ctypes.c_void_p(q.data_ptr()), q.shape[0], q.shape[1], ctypes.byref(desc),
        ctypes.c_void_p(table.data_ptr()), table.shape[1], ctypes.c_void_p(lens.data_ptr()), int(max_len),
        ctypes.c_float(0.0), int(num_splits), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _decode_both(wl, dev, num_splits=0):
    k, v = wl.kv()
    cfg, cache = gpu_store(wl, wl.layers[-1], dev, k, v)
    q = wl.q()
    ref = gpu_decode(wl, cfg, cache, q, dev, num_splits=num_splits)
    table = torch.from_numpy(wl.layout()[0]).to(dev)
    lens = torch.from_numpy(wl.seq_lens.astype(np.int32)).to(dev)
    out = torch.full((wl.num_seqs, wl.num_q_heads, wl.head_dim), float("nan"), dtype=torch.float32, device=dev)
    status = _noalloc_call(cfg, bf16(q, dev), cache, table, lens, int(wl.seq_lens.max()), out, num_splits)
    assert status == 0, tq.lib().tq_last_error().decode()
    torch.cuda.synchronize()
    assert cache.error_flags() == 0
    return out.cpu().numpy(), ref


def test_noalloc_matches_workspace_decode_two_calls(cuda_device):
    # first call: ragged 3-bit-key / 4-bit-value batch with norm correction
    got, ref = _decode_both(W.small("c1", [1, 17, 250, 700]), cuda_device)
    assert_rows_close(got, ref, rtol=DECODE_RTOL)
    # second call, different shapes and format: FP8 keys, a larger split count;
    # the scratch still holds the first call's partials
    got, ref = _decode_both(W.custom(256, 8, 4, False, 2, 16, 48, [200, 1000, 33], 2600), cuda_device,
                            num_splits=9)
    assert_rows_close(got, ref, rtol=DECODE_RTOL)


def test_noalloc_rejects_decode_beyond_scratch(cuda_device):
    wl = W.custom(256, 4, 4, True, 8, 64, 16, [16], 2700)
    cfg = tq.tq_config_init(wl.head_dim, wl.key_bits, wl.value_bits, wl.norm_correction)
    seqs, max_len, splits = 64, 16384, 64
    need = tq.tq_decode_workspace_size(cfg, seqs, 64, 8, 16, max_len, splits)
    assert need > tq.TQ_NOALLOC_SCRATCH_BYTES
    cache = tq.new_paged_cache(cfg, 4, 16, 8, device=cuda_device)
    q = torch.zeros((seqs, 64, 256), dtype=torch.bfloat16, device=cuda_device)
    out = torch.zeros((seqs, 64, 256), dtype=torch.float32, device=cuda_device)
    table = torch.zeros((seqs, 4), dtype=torch.int32, device=cuda_device)
    lens = torch.zeros(seqs, dtype=torch.int32, device=cuda_device)
    status = _noalloc_call(cfg, q, cache, table, lens, max_len, out, splits)
    assert status == 4  # TQ_ERR_WORKSPACE, nothing enqueued
    assert b"no-allocation" in tq.lib().tq_last_error()
    torch.cuda.synchronize()
    assert not out.any()


def test_noalloc_auto_split_count_shrinks_to_fit(cuda_device):
    """With num_splits = 0, a batch whose automatic split count needs more
    partial storage than the scratch holds runs with the most splits that
    fit (here the c4 decode shape: 256 sequences x 16 query heads, d = 256),
    and equals the workspace decode at that split count."""
    wl = W.custom(256, 4, 4, True, 4, 16, 16, [48] * 256, 2800)
    seqs, hq, max_len = 256, 16, 2048
    cfg = tq.tq_config_init(wl.head_dim, wl.key_bits, wl.value_bits, wl.norm_correction)
    auto = tq.tq_decode_workspace_size(cfg, seqs, hq, 4, 16, max_len, 0)
    if auto <= tq.TQ_NOALLOC_SCRATCH_BYTES:
        pytest.skip("the automatic split count fits the scratch on this device")
    fit = tq.TQ_NOALLOC_SCRATCH_BYTES // (seqs * hq * (256 + 2) * 4)
    assert fit >= 1
    k, v = wl.kv()
    cfg, cache = gpu_store(wl, 0, cuda_device, k, v)
    qd = bf16(wl.q(), cuda_device)
    table_np = np.zeros((seqs, max_len // 16), dtype=np.int32)  # room for max_len tokens, 48 used
    table_np[:, :3] = wl.layout()[0]
    table = torch.from_numpy(table_np).to(cuda_device)
    lens = torch.from_numpy(wl.seq_lens.astype(np.int32)).to(cuda_device)
    out = torch.full((seqs, hq, 256), float("nan"), dtype=torch.float32, device=cuda_device)
    status = _noalloc_call(cfg, qd, cache, table, lens, max_len, out, 0)
    assert status == 0, tq.lib().tq_last_error().decode()
    ws = torch.zeros(tq.tq_decode_workspace_size(cfg, seqs, hq, 4, 16, max_len, int(fit)), dtype=torch.uint8,
                     device=cuda_device)
    ref = torch.empty_like(out)
    tq.tq_decode_attention(cfg, qd, cache, table, lens, max_len, ref, ws, num_splits=int(fit))
    torch.cuda.synchronize()
    assert cache.error_flags() == 0
    assert torch.equal(out, ref)
