"""Ring-buffered store and ring decode on the GPU against the oracle.

A prefill and then single-token decode steps go through tq_ring_append on
the GPU and through the oracle's ring_append on the same seeded rows.  The
packed cache follows the store's parity rules (bytes bit-exact outside the
near-boundary exemptions), the ring rows are bit-exact bf16 copies, and
bytes of positions still in the ring stay untouched.  The ring decode runs
on the oracle's own cache and ring, within the decode tolerance.
"""
import numpy as np
import pytest
import torch

import kv_cache_quantization_store_gb300 as tq
import oracle as O
from kv_cache_quantization_store_gb300 import workloads as W
from tq_gpu_util import assert_rows_close, bf16, compare_slots, host_cfg, oracle_layer, slot_bytes, upload_cache

pytestmark = pytest.mark.gpu

PROMPTS = [250, 5, 128]
STEPS = [50, 40, 0]
FINAL = [p + s for p, s in zip(PROMPTS, STEPS)]


def ring_cases():
    return [
        W.custom(128, 3, 4, True, 8, 32, 16, FINAL, 3101, kv_mode="outliers"),
        W.custom(128, 8, 4, False, 8, 32, 16, FINAL, 3102, kv_mode="lognormal"),
        W.custom(64, 4, 3, True, 4, 20, 16, FINAL, 3103),
        W.custom(256, 4, 4, True, 4, 16, 512, FINAL, 3104),
        W.custom(32, 3, 3, False, 2, 2, 32, FINAL, 3105),
    ]


CASES = ring_cases()
IDS = [w.name for w in CASES]


def run_appends(wl, r_len, device, api="append"):
    """The same prefill and decode steps on the GPU and in the oracle; the
    GPU's decode steps go through tq_ring_append or tq_ring_step (api).
    Returns (gpu cache, gpu rings, oracle cache, oracle rings, near dict, cfg, layer)."""
    layer = oracle_layer(wl, 0)
    cfg = host_cfg(wl)
    k_all, v_all = wl.kv()
    cu = wl.cu_seqlens()
    table, nblk = wl.layout()
    n_seq, h_n, d = len(FINAL), wl.num_kv_heads, wl.head_dim
    ocache = O.new_cache(layer.cfg, nblk, wl.block_size, h_n)
    ork = np.zeros((n_seq, r_len, h_n, d), dtype=np.float32)
    orv = np.zeros_like(ork)
    gcache = tq.new_paged_cache(cfg, nblk, wl.block_size, h_n, 0, device=device)
    grk, grv = tq.new_ring(cfg, n_seq, h_n, r_len, device=device)
    gtable = torch.from_numpy(table.astype(np.int32)).to(device)
    ws = torch.empty(tq.tq_ring_workspace_size(n_seq), dtype=torch.uint8, device=device)
    near = {}

    def both(rows, lens):
        counts = [len(r) for r in rows]
        cu_new = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        idx = np.concatenate([np.asarray(r, dtype=np.int64) for r in rows]) if sum(counts) else np.zeros(0, np.int64)
        kn, vn = k_all[idx], v_all[idx]
        near.update(O.ring_append(layer, ocache, table, ork, orv, np.asarray(lens), kn, vn, cu_new))
        kt = bf16(kn, device) if len(idx) else torch.empty((0, h_n, d), dtype=torch.bfloat16, device=device)
        vt = bf16(vn, device) if len(idx) else torch.empty((0, h_n, d), dtype=torch.bfloat16, device=device)
        tq.tq_ring_append(cfg, kt, vt, torch.from_numpy(cu_new).to(device),
                          torch.tensor(lens, dtype=torch.int32, device=device), grk, grv, gcache, gtable, ws)

    def step(rows, lens):
        """One token per sequence through tq_ring_step (idle sequences: seq_lens -1, any row)."""
        cu_new = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
        idx = np.concatenate([np.asarray(r, dtype=np.int64) for r in rows])
        near.update(O.ring_append(layer, ocache, table, ork, orv, np.asarray(lens), k_all[idx], v_all[idx], cu_new))
        one = np.array([r[0] if r else 0 for r in rows], dtype=np.int64)
        tq.tq_ring_step(cfg, bf16(k_all[one], device), bf16(v_all[one], device),
                        torch.tensor(lens, dtype=torch.int32, device=device), grk, grv, gcache, gtable)

    both([range(cu[s], cu[s] + PROMPTS[s]) for s in range(n_seq)], [0] * n_seq)
    for i in range(max(STEPS)):
        rows = [[cu[s] + PROMPTS[s] + i] if i < STEPS[s] else [] for s in range(n_seq)]
        lens = [PROMPTS[s] + i if i < STEPS[s] else -1 for s in range(n_seq)]
        (step if api == "step" else both)(rows, lens)
    torch.cuda.synchronize()
    return gcache, (grk, grv), ocache, (ork, orv), near, cfg, layer


@pytest.mark.parametrize("api", ["append", "step"])
@pytest.mark.parametrize("r_len", [32, 128])
@pytest.mark.parametrize("wl", CASES, ids=IDS)
def test_ring_append_parity(cuda_device, wl, r_len, api):
    gcache, (grk, grv), ocache, (ork, orv), near, cfg, layer = run_appends(wl, r_len, cuda_device, api)
    assert gcache.error_flags() == 0
    k_all, _ = wl.kv()
    cu = wl.cu_seqlens()
    table, _ = wl.layout()
    flat = gcache.data.cpu().numpy()
    slot_al = cfg.slot_size_aligned
    written = np.zeros(flat.shape, dtype=bool)
    for s, n in enumerate(FINAL):
        packed, n_ring = O.ring_split(n, r_len)
        pos = np.arange(packed)
        slots = table[s][pos // wl.block_size].astype(np.int64) * wl.block_size + pos % wl.block_size
        if packed:
            got = slot_bytes(flat, wl, slot_al, slots).reshape(-1, slot_al)
            want = slot_bytes(ocache.data, wl, slot_al, slots).reshape(-1, slot_al)
            nr = np.stack([near[(s, int(p))] for p in pos]).reshape(-1, wl.head_dim)
            compare_slots(layer, got, want, nr, k_all[cu[s]:cu[s] + packed].reshape(-1, wl.head_dim))
            stride = wl.block_size * wl.num_kv_heads * slot_al
            blk, off = np.divmod(slots, wl.block_size)
            base = blk * stride + off * wl.num_kv_heads * slot_al
            written[(base[:, None] + np.arange(wl.num_kv_heads * slot_al)).ravel()] = True
        # ring rows: exact copies of the newest tokens
        got_k = grk[s, :n_ring].float().cpu().numpy()
        got_v = grv[s, :n_ring].float().cpu().numpy()
        np.testing.assert_array_equal(got_k, ork[s, :n_ring])
        np.testing.assert_array_equal(got_v, orv[s, :n_ring])
    assert not flat[~written].any(), "bytes outside the packed positions were written"


@pytest.mark.parametrize("r_len", [32, 128])
@pytest.mark.parametrize("wl", CASES, ids=IDS)
def test_ring_decode_parity(cuda_device, wl, r_len):
    layer = oracle_layer(wl, 0)
    cfg = host_cfg(wl)
    k_all, v_all = wl.kv()
    cu = wl.cu_seqlens()
    table, nblk = wl.layout()
    n_seq, h_n, d = len(FINAL), wl.num_kv_heads, wl.head_dim
    ocache = O.new_cache(layer.cfg, nblk, wl.block_size, h_n)
    ork = np.zeros((n_seq, r_len, h_n, d), dtype=np.float32)
    orv = np.zeros_like(ork)
    O.ring_append(layer, ocache, table, ork, orv, np.zeros(n_seq, dtype=np.int64), k_all, v_all, cu)
    q = wl.q()
    want = O.decode_attention_ring(layer, q, ocache, table, np.asarray(FINAL), ork, orv)
    cache = upload_cache(ocache, cfg, 0, cuda_device)
    gq = bf16(q, cuda_device)
    grk, grv = bf16(ork, cuda_device), bf16(orv, cuda_device)
    gtable = torch.from_numpy(table.astype(np.int32)).to(cuda_device)
    lens = torch.tensor(FINAL, dtype=torch.int32, device=cuda_device)
    for splits in (0, 1, 3):
        ws = torch.zeros(tq.tq_decode_ring_workspace_size(cfg, n_seq, wl.num_q_heads, h_n, wl.block_size,
                                                          max(FINAL), splits), dtype=torch.uint8, device=cuda_device)
        out = torch.empty((n_seq, wl.num_q_heads, d), dtype=torch.float32, device=cuda_device)
        tq.tq_decode_attention_ring(cfg, gq, cache, gtable, lens, max(FINAL), grk, grv, out, ws, num_splits=splits)
        torch.cuda.synchronize()
        assert_rows_close(out.cpu().numpy(), want)
    assert cache.error_flags() == 0


def test_ring_decode_without_ring_tokens_matches_plain_decode(cuda_device):
    """Lengths that are whole ring blocks: the ring decode and the plain
    decode read the same packed tokens and agree to rounding."""
    wl = W.custom(128, 4, 4, True, 8, 32, 16, [256, 128], 3106)
    layer = oracle_layer(wl, 0)
    cfg = host_cfg(wl)
    k_all, v_all = wl.kv()
    ocache = O.new_cache(layer.cfg, wl.layout()[1], wl.block_size, wl.num_kv_heads)
    O.store_kv(layer, k_all, v_all, wl.slot_mapping(), ocache)
    cache = upload_cache(ocache, cfg, 0, cuda_device)
    q = bf16(wl.q(), cuda_device)
    table = torch.from_numpy(wl.layout()[0].astype(np.int32)).to(cuda_device)
    lens = torch.tensor([256, 128], dtype=torch.int32, device=cuda_device)
    grk, grv = tq.new_ring(cfg, 2, wl.num_kv_heads, 128, device=cuda_device)
    ws_r = torch.zeros(tq.tq_decode_ring_workspace_size(cfg, 2, 32, 8, 16, 256, 2), dtype=torch.uint8,
                       device=cuda_device)
    ws = torch.zeros(tq.tq_decode_workspace_size(cfg, 2, 32, 8, 16, 256, 2), dtype=torch.uint8, device=cuda_device)
    o_r = torch.empty((2, 32, 128), dtype=torch.float32, device=cuda_device)
    o_p = torch.empty_like(o_r)
    tq.tq_decode_attention_ring(cfg, q, cache, table, lens, 256, grk, grv, o_r, ws_r, num_splits=2)
    tq.tq_decode_attention(cfg, q, cache, table, lens, 256, o_p, ws, num_splits=2)
    torch.cuda.synchronize()
    np.testing.assert_allclose(o_r.cpu().numpy(), o_p.cpu().numpy(), rtol=0, atol=1e-6)


def test_ring_step_in_cuda_graph(cuda_device):
    """One decode step (ring append, then ring decode, whose ring partial
    forks onto the library's side stream) captured in a CUDA graph gives
    the eager results."""
    wl = W.custom(128, 4, 4, True, 8, 32, 16, [300, 200], 3107)
    cfg = host_cfg(wl)
    k_all, v_all = wl.kv()
    table, nblk = wl.layout()
    cu = wl.cu_seqlens()
    gtable = torch.from_numpy(table.astype(np.int32)).to(cuda_device)
    q = bf16(wl.q(), cuda_device)
    lens_before = torch.tensor([299, 199], dtype=torch.int32, device=cuda_device)
    lens_after = lens_before + 1
    one_each = torch.arange(3, dtype=torch.int32, device=cuda_device)
    k_step = bf16(k_all[[cu[0] + 299, cu[1] + 199]], cuda_device)
    v_step = bf16(v_all[[cu[0] + 299, cu[1] + 199]], cuda_device)
    ws_a = torch.empty(tq.tq_ring_workspace_size(2), dtype=torch.uint8, device=cuda_device)
    ws_d = torch.zeros(tq.tq_decode_ring_workspace_size(cfg, 2, 32, 8, 16, 300), dtype=torch.uint8,
                       device=cuda_device)

    def fresh():
        cache = tq.new_paged_cache(cfg, nblk, 16, 8, 0, device=cuda_device)
        rk, rv = tq.new_ring(cfg, 2, 8, 128, device=cuda_device)
        pre = np.concatenate([np.arange(cu[0], cu[0] + 299), np.arange(cu[1], cu[1] + 199)])
        tq.tq_ring_append(cfg, bf16(k_all[pre], cuda_device), bf16(v_all[pre], cuda_device),
                          torch.tensor([0, 299, 498], dtype=torch.int32, device=cuda_device),
                          torch.zeros(2, dtype=torch.int32, device=cuda_device), rk, rv, cache, gtable, ws_a)
        return cache, rk, rv

    def step(cache, rk, rv, out, stream=None):
        tq.tq_ring_append(cfg, k_step, v_step, one_each, lens_before, rk, rv, cache, gtable, ws_a, stream=stream)
        tq.tq_decode_attention_ring(cfg, q, cache, gtable, lens_after, 300, rk, rv, out, ws_d, stream=stream)

    c1, rk1, rv1 = fresh()
    out_eager = torch.empty((2, 32, 128), dtype=torch.float32, device=cuda_device)
    step(c1, rk1, rv1, out_eager)
    c2, rk2, rv2 = fresh()
    out_graph = torch.full((2, 32, 128), float("nan"), dtype=torch.float32, device=cuda_device)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(c2, rk2, rv2, out_graph)
    g.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out_graph.cpu().numpy(), out_eager.cpu().numpy())
    np.testing.assert_array_equal(c2.data.cpu().numpy(), c1.data.cpu().numpy())
    assert c1.error_flags() == 0 and c2.error_flags() == 0
