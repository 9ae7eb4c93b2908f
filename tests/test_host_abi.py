"""Host-side checks of the C ABI (no GPU): exports, config, signs, errors."""
import ctypes
import re
from pathlib import Path

import numpy as np
import pytest

import oracle as O

HEADER = Path(__file__).resolve().parent.parent / "include" / "tq.h"


def declared_functions():
    text = HEADER.read_text()
    return re.findall(r"^TQ_API\s+[\w\s\*]+?\b(tq_\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_boundary():
    names = set(declared_functions())
    for want in ("tq_config_from_preset", "tq_config_init", "tq_store_kv", "tq_decode_workspace_size",
                 "tq_decode_attention", "tq_dequant", "tq_status_str"):
        assert want in names


def test_library_exports_every_declared_symbol(libtq):
    for name in declared_functions():
        assert hasattr(libtq, name), name


def test_struct_layouts_match_header(tmp_path):
    """The ctypes structs agree with the C compiler's layout of tq.h."""
    import shutil
    import subprocess

    from kv_cache_quantization_store_gb300 import TqCache, TqConfig

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lines = []
    for struct, cls in (("tq_config", TqConfig), ("tq_cache", TqCache)):
        lines.append(f'printf("{struct} size %zu\\n", sizeof({struct}));')
        for name, _ in cls._fields_:
            lines.append(f'printf("{struct} {name} %zu\\n", offsetof({struct}, {name}));')
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "tq.h"\nint main(void) {\n'
                   + "\n".join(lines) + "\nreturn 0; }\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, f"-I{HEADER.parent}", str(src), "-o", str(exe)], check=True)
    got = {}
    for line in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines():
        struct, field, val = line.split()
        got[(struct, field)] = int(val)
    for struct, cls in (("tq_config", TqConfig), ("tq_cache", TqCache)):
        assert got[(struct, "size")] == ctypes.sizeof(cls)
        for name, _ in cls._fields_:
            assert got[(struct, name)] == getattr(cls, name).offset, (struct, name)


@pytest.mark.parametrize("d,kb,vb,nc", [(16, 3, 3, 0), (32, 4, 4, 1), (64, 3, 4, 0), (128, 3, 4, 1),
                                        (128, 8, 4, 0), (128, 3, 3, 1), (256, 4, 4, 1), (256, 8, 3, 0)])
def test_host_config_matches_oracle(libtq, d, kb, vb, nc):
    from kv_cache_quantization_store_gb300 import tq_config_init

    h = tq_config_init(d, kb, vb, bool(nc), seed=42)
    o = O.Config(head_dim=d, key_quant_bits=kb, value_quant_bits=vb, norm_correction=bool(nc))
    assert (h.key_fp8, h.mse_bits, h.key_mse_bits, h.n_centroids) == (o.key_fp8, o.mse_bits, o.key_mse_bits,
                                                                      o.n_centroids)
    assert (h.key_packed_size, h.value_packed_size, h.slot_size, h.slot_size_aligned) == (
        o.key_packed_size, o.value_packed_size, o.slot_size, o.slot_size_aligned)
    cb = O.codebook(d, o.mse_bits)
    np.testing.assert_array_equal(np.array(h.centroid_list(), dtype=np.float32), cb.centroids)
    np.testing.assert_array_equal(np.array(h.boundary_list(), dtype=np.float32), cb.boundaries)
    assert 0 < h.lloyd_max_iterations < 100000


def test_presets(libtq):
    from kv_cache_quantization_store_gb300 import PRESETS, tq_config_from_preset

    assert set(PRESETS) == set(O.PRESETS)
    for name in PRESETS:
        h = tq_config_from_preset(128, name)
        o = O.config_from_preset(name, 128)
        assert (h.key_quant_bits, h.value_quant_bits, bool(h.norm_correction), h.seed) == (
            o.key_quant_bits, o.value_quant_bits, o.norm_correction, o.seed)
        assert h.slot_size_aligned == o.slot_size_aligned


def test_unknown_preset_error(libtq):
    from kv_cache_quantization_store_gb300 import TQError, tq_config_from_preset

    with pytest.raises(TQError) as e:
        tq_config_from_preset(128, "turboquant_k2v2")
    assert e.value.status == 2
    for name in O.PRESETS:
        assert name in str(e.value)


@pytest.mark.parametrize("args,status", [((96, 3, 4), 3), ((8, 3, 4), 3), ((0, 3, 4), 1), ((128, 2, 4), 1),
                                         ((128, 5, 4), 1), ((128, 3, 2), 1), ((128, 3, 8), 1)])
def test_config_rejects(libtq, args, status):
    from kv_cache_quantization_store_gb300 import TQError, tq_config_init

    with pytest.raises(TQError) as e:
        tq_config_init(*args)
    assert e.value.status == status


@pytest.mark.parametrize("d", [16, 64, 128, 256])
def test_signs_match_oracle(libtq, d):
    from kv_cache_quantization_store_gb300 import tq_config_init, tq_layer_signs

    cfg = tq_config_init(d, 3, 4)
    for layer in (0, 1, 3, 17):
        np.testing.assert_array_equal(np.array(tq_layer_signs(cfg, layer)),
                                      O.random_signs(O.layer_seed(42, layer), d))


def test_hybrid_page(libtq):
    from kv_cache_quantization_store_gb300 import tq_config_from_preset, tq_hybrid_page

    cfg = tq_config_from_preset(256, "turboquant_4bit_nc")
    assert tq_hybrid_page(cfg, 4, 2) == (536576, 512)
    assert tq_hybrid_page(cfg, 4, 0) == (1048, 1)
    cfg = tq_config_from_preset(128, "turboquant_k3v4_nc")
    page, tok = tq_hybrid_page(cfg, 8, 2)
    assert page == O.hybrid_page_bytes(8 * 118, 2 * 8 * 128 * 2) and tok * 8 * 118 == page


def _cache(data=16, num_blocks=4, block_size=16, heads=1, stride=0):
    from kv_cache_quantization_store_gb300 import TqCache

    return TqCache(data, num_blocks, block_size, heads, 0, 0, stride, None)


def test_store_argument_errors(libtq):
    from kv_cache_quantization_store_gb300 import tq_config_init

    cfg = tq_config_init(64, 3, 4)
    c = _cache()
    call = lambda k, v, n, sm, cache: libtq.tq_store_kv(ctypes.byref(cfg), k, v, n, sm, ctypes.byref(cache), None)
    assert call(None, None, 0, None, c) == 0                       # nothing to do
    assert call(None, 64, 4, 64, c) == 1                            # null k
    assert call(64, 64, -1, 64, c) == 1                             # negative count
    assert call(64 + 2, 64, 4, 64, c) == 1                          # misaligned k
    assert call(64, 64, 4, 64, _cache(data=None)) == 1              # null cache
    assert call(64, 64, 4, 64, _cache(stride=16)) == 1              # stride < block
    assert call(64, 64, 4, 64, _cache(data=17)) == 1                # odd cache address
    bad = tq_config_init(64, 3, 4)
    bad.slot_size_aligned += 2
    assert libtq.tq_store_kv(ctypes.byref(bad), 64, 64, 4, 64, ctypes.byref(c), None) == 1
    assert b"match" in libtq.tq_last_error()


def test_decode_argument_errors(libtq):
    from kv_cache_quantization_store_gb300 import tq_config_init

    cfg = tq_config_init(64, 3, 4)

    def call(cache, hq=2, ws=1 << 20):
        return libtq.tq_decode_attention(ctypes.byref(cfg), 64, 1, hq, ctypes.byref(cache), 64, 4, 64, 64, 0.0,
                                         0, 64, 64, ws, None)

    assert call(_cache(heads=2), hq=3) == 1          # Hq not a multiple of H
    assert call(_cache(data=24)) == 1                # cache not 16-byte aligned
    assert call(_cache(block_size=8)) == 3           # block size not a multiple of 16
    assert call(_cache(heads=16), hq=16) == 3        # more KV heads than built
    assert call(_cache(heads=1), hq=16) == 3         # GQA group above 8


def test_sequence_limit(libtq):
    """Decode and dequant take one grid row per sequence: above TQ_MAX_SEQS
    they return TQ_ERR_UNSUPPORTED before anything is enqueued; at the limit
    the next check (a NULL pointer here) answers."""
    from kv_cache_quantization_store_gb300 import TQ_MAX_SEQS, tq_config_init

    text = HEADER.read_text()
    assert int(re.search(r"#define TQ_MAX_SEQS (\d+)", text).group(1)) == TQ_MAX_SEQS == 65535
    cfg = tq_config_init(64, 3, 4)
    c = _cache()

    def decode(seqs, q=64):
        return libtq.tq_decode_attention(ctypes.byref(cfg), q, seqs, 2, ctypes.byref(c), 64, 4, 64, 64, 0.0,
                                         0, 64, 64, 1 << 20, None)

    def ring_decode(seqs, q=64):
        return libtq.tq_decode_attention_ring(ctypes.byref(cfg), q, seqs, 2, ctypes.byref(c), 64, 4, 64, 64, 0.0,
                                              0, 64, 64, 128, 64, 64, 1 << 20, None)

    def dequant(seqs, k=64):
        return libtq.tq_dequant(ctypes.byref(cfg), ctypes.byref(c), 64, 4, 64, seqs, 16, k, 64, None)

    for fn in (decode, ring_decode, dequant):
        assert fn(TQ_MAX_SEQS + 1) == 3, fn.__name__
        assert b"65535" in libtq.tq_last_error()
        assert fn(TQ_MAX_SEQS, None) == 1, fn.__name__


def test_status_strings(libtq):
    from kv_cache_quantization_store_gb300 import tq_status_str

    assert [tq_status_str(i) for i in range(7)] == [
        "TQ_OK", "TQ_ERR_INVALID_ARG", "TQ_ERR_UNKNOWN_PRESET", "TQ_ERR_UNSUPPORTED", "TQ_ERR_WORKSPACE",
        "TQ_ERR_OUT_OF_RANGE", "TQ_ERR_CUDA"]


def test_ring_argument_errors(libtq):
    """tq_ring_append and tq_decode_attention_ring reject bad arguments
    before anything is enqueued (status codes of tq_status)."""
    from kv_cache_quantization_store_gb300 import tq_config_init

    cfg = tq_config_init(64, 3, 4)

    def append(k=64, v=64, n=1, cu=64, seqs=1, lens=64, rk=64, rv=64, r_len=128, cache=None, bt=64, mb=4, ws=64,
               ws_bytes=1 << 10):
        cache = cache or _cache()
        return libtq.tq_ring_append(ctypes.byref(cfg), k, v, n, cu, seqs, lens, rk, rv, r_len, ctypes.byref(cache),
                                    bt, mb, ws, ws_bytes, None)

    assert append(seqs=0) == 0          # no sequences: nothing to do
    assert append(r_len=0) == 3         # ring length outside [1, 128]
    assert append(r_len=129) == 3
    assert append(n=-1) == 1            # negative token count
    assert append(mb=0) == 1            # no block-table columns
    assert append(rk=None) == 1         # missing ring
    assert append(k=None) == 1          # new tokens without rows
    assert append(rk=72) == 1           # ring not 16-byte aligned
    assert append(cu=66) == 1           # cu_new not 4-byte aligned
    assert append(ws=None) == 4         # missing workspace
    assert append(ws_bytes=8) == 4      # workspace too small
    assert append(ws=72) == 4           # workspace not 16-byte aligned
    assert libtq.tq_ring_workspace_size(-1) == 0
    assert libtq.tq_ring_workspace_size(4) >= 5 * 8

    def step(k=64, v=64, seqs=1, lens=64, rk=64, rv=64, r_len=128, bt=64, mb=4):
        return libtq.tq_ring_step(ctypes.byref(cfg), k, v, seqs, lens, rk, rv, r_len, ctypes.byref(_cache()), bt, mb,
                                  None)

    assert step(seqs=0) == 0
    assert step(r_len=0) == 3
    assert step(seqs=-1) == 1
    assert step(k=None) == 1
    assert step(rv=80 + 8) == 1         # ring not 16-byte aligned
    assert step(lens=66) == 1           # seq_lens not 4-byte aligned

    def decode(r_len=128, rk=64, rv=64, hq=2, heads=1):
        return libtq.tq_decode_attention_ring(ctypes.byref(cfg), 64, 1, hq, ctypes.byref(_cache(heads=heads)), 64, 4,
                                              64, 64, 0.0, 0, rk, rv, r_len, 64, 64, 1 << 20, None)

    assert decode(r_len=0) == 3
    assert decode(r_len=200) == 3
    assert decode(rk=None) == 1
    assert decode(rv=72) == 1           # ring not 16-byte aligned
    assert decode(hq=16) == 3           # GQA group above 8


def test_ring_decode_workspace_has_one_more_partial(libtq):
    """The ring decode's workspace holds the splits' partial states plus one
    for the ring rows: S * Hq * (splits + 1) * (d + 2) fp32, in 256-byte units."""
    from kv_cache_quantization_store_gb300 import tq_config_init

    cfg = tq_config_init(64, 3, 4)
    s, hq, h, splits = 2, 8, 4, 3
    plain = libtq.tq_decode_workspace_size(ctypes.byref(cfg), s, hq, h, 16, 1000, splits)
    ring = libtq.tq_decode_ring_workspace_size(ctypes.byref(cfg), s, hq, h, 16, 1000, splits)
    up = lambda x: -(-x // 256) * 256
    assert plain == up(s * hq * splits * 66 * 4)
    assert ring == up(s * hq * (splits + 1) * 66 * 4)


def test_binding_checks_row_shapes(libtq):
    """The binding rejects K/V rows whose trailing dims are not the cache's
    (num_kv_heads, head_dim) before anything reaches the library: the
    kernels index those rows with the cache's H and the config's d."""
    import torch

    import kv_cache_quantization_store_gb300 as tq

    cfg = tq.tq_config_init(64, 3, 4)
    cache = tq.new_paged_cache(cfg, 2, 16, 2, 0, device="cpu", with_flags=False)
    table = torch.zeros((1, 2), dtype=torch.int32)
    cu = torch.tensor([0, 4], dtype=torch.int32)
    lens = torch.zeros(1, dtype=torch.int32)
    rows = lambda *shape: torch.zeros(shape, dtype=torch.bfloat16)

    with pytest.raises(ValueError, match="k_out"):
        tq.tq_dequant(cfg, cache, table, cu, 4, rows(4, 2 * 64), rows(4, 2 * 64))    # flattened rows
    with pytest.raises(ValueError, match="k_out"):
        tq.tq_dequant(cfg, cache, table, cu, 4, rows(4, 1, 64), rows(4, 1, 64))      # wrong head count
    with pytest.raises(ValueError, match="same shape"):
        tq.tq_dequant(cfg, cache, table, cu, 4, rows(4, 2, 64), rows(3, 2, 64))
    ring_ok, ring_bad = rows(1, 8, 2, 64), rows(1, 8, 2, 32)
    with pytest.raises(ValueError, match="ring_k"):
        tq.tq_ring_step(cfg, rows(1, 2, 64), rows(1, 2, 64), lens, ring_bad, ring_bad, cache, table)
    with pytest.raises(ValueError, match="k must be"):
        tq.tq_ring_step(cfg, rows(1, 4, 32), rows(1, 4, 32), lens, ring_ok, ring_ok, cache, table)
    with pytest.raises(ValueError, match="k must be"):
        tq.tq_ring_append(cfg, rows(3, 2, 32), rows(3, 2, 32), cu, lens, ring_ok, ring_ok, cache, table,
                          torch.zeros(64, dtype=torch.uint8))
    q, out = rows(1, 4, 64), torch.zeros((1, 4, 64), dtype=torch.float32)
    with pytest.raises(ValueError, match="ring_k"):
        tq.tq_decode_attention_ring(cfg, q, cache, table, lens, 16, ring_bad, ring_bad, out,
                                    torch.zeros(64, dtype=torch.uint8))


@pytest.mark.parametrize("d", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("bits", [3, 4])
def test_store_bucket_table_has_one_boundary_per_bucket(libtq, d, bits):
    """The store finds a key index through 256 buckets g(y) = RN(127 y + 128 +
    1.5 * 2^23) & 0xFF of the unit-vector coordinate (one fma, tq_store.cu);
    its table holds one boundary per bucket, so every supported codebook's
    fp32 boundaries must fall in distinct buckets, in order."""
    import kv_cache_quantization_store_gb300 as tq

    cfg = tq.tq_config_init(d, bits, 4, False)
    b = np.array(cfg.boundary_list(), dtype=np.float32).astype(np.float64)
    # the fma: exact product and sum in fp64, one rounding to fp32
    g = (b * 127.0 + 12583040.0).astype(np.float32).view(np.uint32) & 0xFF
    assert len(set(g.tolist())) == len(g)
    assert np.all(np.diff(g.astype(np.int64)) > 0)
    assert g.min() >= 1 and g.max() <= 254  # |y| <= 1 maps into [1, 255]
