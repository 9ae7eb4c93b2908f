"""TurboQuant KV-cache store and fused decode attention for GB300 (sm_103a).

A thin ctypes binding over ``libtq.so``, whose C ABI is declared in
``include/tq.h``.  The functions keep the C names.  They only marshal
arguments: they check dtypes, devices and contiguity, pass raw device
pointers and the current torch CUDA stream, and raise ``TQError`` on a non-OK
status.  All computation runs in the library's CUDA kernels.  There is no CPU
fallback: if ``libtq.so`` is missing, the first call fails and says how to
build it.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from pathlib import Path

import torch

__all__ = [
    "TQError", "TqConfig", "TqCache", "PagedCache", "lib", "library_path",
    "tq_config_init", "tq_config_from_preset", "tq_layer_signs", "tq_store_kv",
    "tq_decode_workspace_size", "tq_decode_attention", "tq_decode_attention_noalloc", "tq_dequant",
    "tq_ring_workspace_size", "tq_ring_append", "tq_ring_step", "tq_decode_ring_workspace_size",
    "tq_decode_attention_ring", "tq_dense_decode_workspace_size", "tq_dense_decode_attention",
    "new_ring", "tq_status_str", "TQ_NOALLOC_SCRATCH_BYTES", "TQ_RING_TOKENS", "TQ_MAX_SEQS",
    "new_paged_cache", "tq_hybrid_page", "PRESETS",
]

PRESETS = ("turboquant_k8v4", "turboquant_4bit_nc", "turboquant_k3v4_nc", "turboquant_3bit_nc")

TQ_OK = 0
TQ_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024  # include/tq.h
TQ_FLAG_SLOT_OUT_OF_RANGE = 1
TQ_FLAG_BLOCK_OUT_OF_RANGE = 2
TQ_FLAG_SEQ_TOO_LONG = 4
TQ_FLAG_WAIT_TIMEOUT = 8
TQ_RING_TOKENS = 128  # include/tq.h
TQ_MAX_SEQS = 65535  # include/tq.h: sequences of one decode or dequant call

_PKG = Path(__file__).resolve().parent


def library_path() -> Path:
    return _PKG / "libtq.so"


class TqConfig(ctypes.Structure):
    _fields_ = [
        ("head_dim", ctypes.c_int32),
        ("key_quant_bits", ctypes.c_int32),
        ("value_quant_bits", ctypes.c_int32),
        ("norm_correction", ctypes.c_int32),
        ("seed", ctypes.c_uint64),
        ("key_fp8", ctypes.c_int32),
        ("mse_bits", ctypes.c_int32),
        ("key_mse_bits", ctypes.c_int32),
        ("n_centroids", ctypes.c_int32),
        ("key_packed_size", ctypes.c_int32),
        ("value_packed_size", ctypes.c_int32),
        ("slot_size", ctypes.c_int32),
        ("slot_size_aligned", ctypes.c_int32),
        ("centroids", ctypes.c_float * 16),
        ("boundaries", ctypes.c_float * 15),
        ("lloyd_max_iterations", ctypes.c_int32),
    ]

    def centroid_list(self):
        return list(self.centroids)[: self.n_centroids]

    def boundary_list(self):
        return list(self.boundaries)[: self.n_centroids - 1]


class TqCache(ctypes.Structure):
    _fields_ = [
        ("data_dev", ctypes.c_void_p),
        ("num_blocks", ctypes.c_int64),
        ("block_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("layer_idx", ctypes.c_int32),
        ("reserved0", ctypes.c_int32),
        ("block_stride_bytes", ctypes.c_int64),
        ("error_flags_dev", ctypes.c_void_p),
    ]


class TQError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{tq_status_str(status)}: {message}")
        self.status = status


_LIB = None

_SIGNATURES = {
    "tq_config_init": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_uint64, ctypes.POINTER(TqConfig)]),
    "tq_config_from_preset": (ctypes.c_int, [ctypes.c_int32, ctypes.c_char_p, ctypes.POINTER(TqConfig)]),
    "tq_layer_signs": (ctypes.c_int, [ctypes.POINTER(TqConfig), ctypes.c_int32, ctypes.POINTER(ctypes.c_int8)]),
    "tq_store_kv": (ctypes.c_int, [ctypes.POINTER(TqConfig), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                   ctypes.c_void_p, ctypes.POINTER(TqCache), ctypes.c_void_p]),
    "tq_decode_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(TqConfig), ctypes.c_int32, ctypes.c_int32,
                                                   ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                   ctypes.c_int32]),
    "tq_decode_attention": (ctypes.c_int, [ctypes.POINTER(TqConfig), ctypes.c_void_p, ctypes.c_int32,
                                           ctypes.c_int32, ctypes.POINTER(TqCache), ctypes.c_void_p,
                                           ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_float,
                                           ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                           ctypes.c_void_p]),
    "tq_dequant": (ctypes.c_int, [ctypes.POINTER(TqConfig), ctypes.POINTER(TqCache), ctypes.c_void_p,
                                  ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "tq_decode_attention_noalloc": (ctypes.c_int, [ctypes.POINTER(TqConfig), ctypes.c_void_p, ctypes.c_int32,
                                                   ctypes.c_int32, ctypes.POINTER(TqCache), ctypes.c_void_p,
                                                   ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32,
                                                   ctypes.c_float, ctypes.c_int32, ctypes.c_void_p,
                                                   ctypes.c_void_p]),
    "tq_ring_workspace_size": (ctypes.c_size_t, [ctypes.c_int32]),
    "tq_ring_append": (ctypes.c_int, [ctypes.POINTER(TqConfig), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                      ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(TqCache), ctypes.c_void_p,
                                      ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "tq_ring_step": (ctypes.c_int, [ctypes.POINTER(TqConfig), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                    ctypes.POINTER(TqCache), ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]),
    "tq_decode_ring_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(TqConfig), ctypes.c_int32, ctypes.c_int32,
                                                        ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                        ctypes.c_int32]),
    "tq_decode_attention_ring": (ctypes.c_int, [ctypes.POINTER(TqConfig), ctypes.c_void_p, ctypes.c_int32,
                                                ctypes.c_int32, ctypes.POINTER(TqCache), ctypes.c_void_p,
                                                ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_float,
                                                ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                                ctypes.c_void_p]),
    "tq_dense_decode_workspace_size": (ctypes.c_size_t, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                         ctypes.c_int32, ctypes.c_int32]),
    "tq_dense_decode_attention": (ctypes.c_int, [ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                                 ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                 ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                                                 ctypes.c_size_t, ctypes.c_void_p]),
    "tq_hybrid_page": (ctypes.c_int, [ctypes.POINTER(TqConfig), ctypes.c_int32, ctypes.c_int32,
                                      ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32)]),
    "tq_status_str": (ctypes.c_char_p, [ctypes.c_int]),
    "tq_last_error": (ctypes.c_char_p, []),
}


def lib() -> ctypes.CDLL:
    """Loads libtq.so (built in-tree by ``build.build()``); raises if absent."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not path.exists():
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m kv_cache_quantization_store_gb300.build`")
        handle = ctypes.CDLL(str(path))
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = handle
    return _LIB


def tq_status_str(status: int) -> str:
    return lib().tq_status_str(status).decode()


def _check(status: int):
    if status != TQ_OK:
        raise TQError(status, lib().tq_last_error().decode())


# -- config ------------------------------------------------------------------

def tq_config_init(head_dim: int, key_quant_bits: int, value_quant_bits: int,
                   norm_correction: bool = False, seed: int = 42) -> TqConfig:
    cfg = TqConfig()
    _check(lib().tq_config_init(head_dim, key_quant_bits, value_quant_bits, int(bool(norm_correction)),
                                seed, ctypes.byref(cfg)))
    return cfg


def tq_config_from_preset(head_dim: int, preset: str) -> TqConfig:
    cfg = TqConfig()
    _check(lib().tq_config_from_preset(head_dim, preset.encode(), ctypes.byref(cfg)))
    return cfg


def tq_layer_signs(cfg: TqConfig, layer_idx: int) -> list[int]:
    buf = (ctypes.c_int8 * cfg.head_dim)()
    _check(lib().tq_layer_signs(ctypes.byref(cfg), layer_idx, buf))
    return list(buf)


# -- cache -------------------------------------------------------------------

@dataclass
class PagedCache:
    """A layer's paged byte cache in device memory plus its geometry."""

    data: torch.Tensor          # uint8, num_blocks * block_stride bytes
    num_blocks: int
    block_size: int
    num_kv_heads: int
    layer_idx: int
    block_stride: int
    flags: torch.Tensor | None = None  # int32 [1], kernels OR error bits into it

    def descriptor(self) -> TqCache:
        return TqCache(self.data.data_ptr(), self.num_blocks, self.block_size, self.num_kv_heads,
                       self.layer_idx, 0, self.block_stride,
                       self.flags.data_ptr() if self.flags is not None else None)

    def error_flags(self) -> int:
        return int(self.flags.item()) if self.flags is not None else 0


def new_paged_cache(cfg: TqConfig, num_blocks: int, block_size: int, num_kv_heads: int, layer_idx: int = 0,
                    block_stride: int | None = None, device="cuda", with_flags: bool = True) -> PagedCache:
    """Allocates a zeroed cache of num_blocks blocks (torch device memory)."""
    dense = block_size * num_kv_heads * cfg.slot_size_aligned
    stride = dense if block_stride is None else int(block_stride)
    data = torch.zeros(num_blocks * stride, dtype=torch.uint8, device=device)
    flags = torch.zeros(1, dtype=torch.int32, device=device) if with_flags else None
    return PagedCache(data, num_blocks, block_size, num_kv_heads, layer_idx, stride, flags)


def tq_hybrid_page(cfg: TqConfig, num_kv_heads: int, skip_dtype_bytes: int = 2):
    """(unified page bytes, TQ tokens per page) of a TQ layer in a hybrid
    model; see tq_hybrid_page in include/tq.h."""
    page = ctypes.c_int64()
    tokens = ctypes.c_int32()
    _check(lib().tq_hybrid_page(ctypes.byref(cfg), num_kv_heads, skip_dtype_bytes, ctypes.byref(page),
                                ctypes.byref(tokens)))
    return page.value, tokens.value


# -- kernels -----------------------------------------------------------------

def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dev(t: torch.Tensor, dtype, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _token_rows(t: torch.Tensor, name: str, heads: int, d: int, ring: bool = False):
    """Shape check of K/V rows: [T, H, d], or [S, R, H, d] for a ring.  The
    kernels index these rows with the cache's H and the config's d."""
    want = 4 if ring else 3
    if t.dim() != want or tuple(t.shape[-2:]) != (heads, d):
        lead = "[S, R, " if ring else "["
        raise ValueError(f"{name} must be {lead}num_kv_heads={heads}, head_dim={d}], got {tuple(t.shape)}")


def tq_store_kv(cfg: TqConfig, k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                cache: PagedCache, stream=None):
    """k, v: bf16 [T, H, d]; slot_mapping: int64 [T] (negative = skip)."""
    if k.shape != v.shape or k.dim() != 3 or k.shape[1] != cache.num_kv_heads or k.shape[2] != cfg.head_dim:
        raise ValueError("k and v must both be [T, num_kv_heads, head_dim]")
    if slot_mapping.shape != (k.shape[0],):
        raise ValueError("slot_mapping must be [T]")
    desc = cache.descriptor()
    _check(lib().tq_store_kv(ctypes.byref(cfg), _dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"),
                             k.shape[0], _dev(slot_mapping, torch.int64, "slot_mapping"), ctypes.byref(desc),
                             _stream(stream)))


def tq_decode_workspace_size(cfg: TqConfig, num_seqs: int, num_q_heads: int, num_kv_heads: int,
                             block_size: int, max_seq_len: int, num_splits: int = 0) -> int:
    n = lib().tq_decode_workspace_size(ctypes.byref(cfg), num_seqs, num_q_heads, num_kv_heads, block_size,
                                       max_seq_len, num_splits)
    if n == 0:
        raise TQError(1, "invalid decode workspace query")
    return int(n)


def tq_decode_attention(cfg: TqConfig, q: torch.Tensor, cache: PagedCache, block_table: torch.Tensor,
                        seq_lens: torch.Tensor, max_seq_len: int, out: torch.Tensor, workspace: torch.Tensor,
                        sm_scale: float = 0.0, num_splits: int = 0, stream=None):
    """q: bf16 [S, Hq, d]; block_table int32 [S, max_blocks]; seq_lens int32 [S];
    out: fp32 [S, Hq, d]; workspace: zero-initialised uint8 device buffer."""
    if q.dim() != 3 or q.shape[2] != cfg.head_dim:
        raise ValueError("q must be [num_seqs, num_q_heads, head_dim]")
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if block_table.dim() != 2 or block_table.shape[0] != q.shape[0] or seq_lens.shape != (q.shape[0],):
        raise ValueError("block_table must be [S, max_blocks] and seq_lens [S]")
    desc = cache.descriptor()
    _check(lib().tq_decode_attention(
        ctypes.byref(cfg), _dev(q, torch.bfloat16, "q"), q.shape[0], q.shape[1], ctypes.byref(desc),
        _dev(block_table, torch.int32, "block_table"), block_table.shape[1],
        _dev(seq_lens, torch.int32, "seq_lens"), int(max_seq_len), float(sm_scale), int(num_splits),
        _dev(out, torch.float32, "out"), _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
        _stream(stream)))


def tq_decode_attention_noalloc(cfg: TqConfig, q: torch.Tensor, cache: PagedCache, block_table: torch.Tensor,
                                seq_lens: torch.Tensor, max_seq_len: int, out: torch.Tensor, sm_scale: float = 0.0,
                                num_splits: int = 0, stream=None):
    """tq_decode_attention without a workspace argument, for callers that
    cannot allocate device memory: it runs on the library's fixed static
    scratch (see tq_decode_attention_noalloc in include/tq.h for the size
    limit and why overlapping calls race)."""
    if q.dim() != 3 or q.shape[2] != cfg.head_dim or out.shape != q.shape:
        raise ValueError("q and out must be [num_seqs, num_q_heads, head_dim]")
    if block_table.dim() != 2 or block_table.shape[0] != q.shape[0] or seq_lens.shape != (q.shape[0],):
        raise ValueError("block_table must be [S, max_blocks] and seq_lens [S]")
    desc = cache.descriptor()
    _check(lib().tq_decode_attention_noalloc(
        ctypes.byref(cfg), _dev(q, torch.bfloat16, "q"), q.shape[0], q.shape[1], ctypes.byref(desc),
        _dev(block_table, torch.int32, "block_table"), block_table.shape[1],
        _dev(seq_lens, torch.int32, "seq_lens"), int(max_seq_len), float(sm_scale), int(num_splits),
        _dev(out, torch.float32, "out"), _stream(stream)))


# -- dequant-then-dense comparison path ([ART] article, "Obstacle 1") -------------------

def tq_dense_decode_workspace_size(head_dim: int, num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                   max_seq_len: int) -> int:
    n = lib().tq_dense_decode_workspace_size(head_dim, num_seqs, num_q_heads, num_kv_heads, max_seq_len)
    if n == 0:
        raise TQError(1, "invalid dense decode workspace query")
    return int(n)


def tq_dense_decode_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens: torch.Tensor,
                              max_seq_len: int, out: torch.Tensor, workspace: torch.Tensor, sm_scale: float = 0.0,
                              stream=None):
    """Attention over bf16 K/V rows (the layout tq_dequant writes): q bf16
    [S, Hq, d]; k, v bf16 [rows, H, d]; cu_seqlens int32 [S + 1]; out fp32
    [S, Hq, d]; workspace uint8, tq_dense_decode_workspace_size bytes."""
    if q.dim() != 3 or k.dim() != 3 or v.shape != k.shape or k.shape[2] != q.shape[2] or out.shape != q.shape:
        raise ValueError("q and out must be [S, Hq, d], k and v [rows, H, d]")
    if cu_seqlens.shape != (q.shape[0] + 1,):
        raise ValueError("cu_seqlens must be [num_seqs + 1]")
    _check(lib().tq_dense_decode_attention(
        q.shape[2], _dev(q, torch.bfloat16, "q"), q.shape[0], q.shape[1], k.shape[1], _dev(k, torch.bfloat16, "k"),
        _dev(v, torch.bfloat16, "v"), _dev(cu_seqlens, torch.int32, "cu_seqlens"), int(max_seq_len),
        float(sm_scale), _dev(out, torch.float32, "out"), _dev(workspace, torch.uint8, "workspace"),
        workspace.numel(), _stream(stream)))


# -- ring-buffered store ([ART] article, full_tq write path) ------------------------

def new_ring(cfg: TqConfig, num_seqs: int, num_kv_heads: int, ring_tokens: int = TQ_RING_TOKENS,
             device="cuda"):
    """(ring_k, ring_v): bf16 [num_seqs, ring_tokens, num_kv_heads, head_dim]."""
    shape = (num_seqs, ring_tokens, num_kv_heads, cfg.head_dim)
    return (torch.zeros(shape, dtype=torch.bfloat16, device=device),
            torch.zeros(shape, dtype=torch.bfloat16, device=device))


def tq_ring_workspace_size(num_seqs: int) -> int:
    return int(lib().tq_ring_workspace_size(num_seqs))


def tq_ring_append(cfg: TqConfig, k: torch.Tensor, v: torch.Tensor, cu_new: torch.Tensor, seq_lens: torch.Tensor,
                   ring_k: torch.Tensor, ring_v: torch.Tensor, cache: PagedCache, block_table: torch.Tensor,
                   workspace: torch.Tensor, stream=None):
    """k, v: bf16 [T, H, d] new tokens, sequence s's rows cu_new[s]..cu_new[s+1]-1
    (int32 [S + 1]); seq_lens int32 [S]: tokens before the call; rings from new_ring."""
    num_seqs = seq_lens.shape[0]
    if cu_new.shape != (num_seqs + 1,) or block_table.dim() != 2 or block_table.shape[0] != num_seqs:
        raise ValueError("cu_new must be [S + 1] and block_table [S, max_blocks]")
    if ring_k.shape != ring_v.shape or ring_k.dim() != 4 or ring_k.shape[0] != num_seqs:
        raise ValueError("ring_k and ring_v must be [S, R, H, d]")
    _token_rows(ring_k, "ring_k", cache.num_kv_heads, cfg.head_dim, ring=True)
    if k.shape != v.shape:
        raise ValueError("k and v must have the same shape")
    _token_rows(k, "k", cache.num_kv_heads, cfg.head_dim)
    desc = cache.descriptor()
    _check(lib().tq_ring_append(
        ctypes.byref(cfg), _dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"), k.shape[0],
        _dev(cu_new, torch.int32, "cu_new"), num_seqs, _dev(seq_lens, torch.int32, "seq_lens"),
        _dev(ring_k, torch.bfloat16, "ring_k"), _dev(ring_v, torch.bfloat16, "ring_v"), ring_k.shape[1],
        ctypes.byref(desc), _dev(block_table, torch.int32, "block_table"), block_table.shape[1],
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)))


def tq_ring_step(cfg: TqConfig, k: torch.Tensor, v: torch.Tensor, seq_lens: torch.Tensor, ring_k: torch.Tensor,
                 ring_v: torch.Tensor, cache: PagedCache, block_table: torch.Tensor, stream=None):
    """One decode step, one new token per sequence: k, v bf16 [S, H, d];
    seq_lens int32 [S], tokens before the step (tq_ring_step in include/tq.h)."""
    num_seqs = seq_lens.shape[0]
    if k.dim() != 3 or k.shape[0] != num_seqs or v.shape != k.shape:
        raise ValueError("k and v must be [S, H, d] with one row per sequence")
    _token_rows(k, "k", cache.num_kv_heads, cfg.head_dim)
    if block_table.dim() != 2 or block_table.shape[0] != num_seqs:
        raise ValueError("block_table must be [S, max_blocks]")
    if ring_k.shape != ring_v.shape or ring_k.dim() != 4 or ring_k.shape[0] != num_seqs:
        raise ValueError("ring_k and ring_v must be [S, R, H, d]")
    _token_rows(ring_k, "ring_k", cache.num_kv_heads, cfg.head_dim, ring=True)
    desc = cache.descriptor()
    _check(lib().tq_ring_step(
        ctypes.byref(cfg), _dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"), num_seqs,
        _dev(seq_lens, torch.int32, "seq_lens"), _dev(ring_k, torch.bfloat16, "ring_k"),
        _dev(ring_v, torch.bfloat16, "ring_v"), ring_k.shape[1], ctypes.byref(desc),
        _dev(block_table, torch.int32, "block_table"), block_table.shape[1], _stream(stream)))


def tq_decode_ring_workspace_size(cfg: TqConfig, num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                  block_size: int, max_seq_len: int, num_splits: int = 0) -> int:
    n = lib().tq_decode_ring_workspace_size(ctypes.byref(cfg), num_seqs, num_q_heads, num_kv_heads, block_size,
                                            max_seq_len, num_splits)
    if n == 0:
        raise TQError(1, "invalid decode sizes")
    return int(n)


def tq_decode_attention_ring(cfg: TqConfig, q: torch.Tensor, cache: PagedCache, block_table: torch.Tensor,
                             seq_lens: torch.Tensor, max_seq_len: int, ring_k: torch.Tensor, ring_v: torch.Tensor,
                             out: torch.Tensor, workspace: torch.Tensor, sm_scale: float = 0.0, num_splits: int = 0,
                             stream=None):
    """Decode over the packed whole ring blocks plus the exact ring rows;
    seq_lens counts both (tq_decode_attention_ring in include/tq.h)."""
    if q.dim() != 3 or q.shape[2] != cfg.head_dim or out.shape != q.shape:
        raise ValueError("q and out must be [num_seqs, num_q_heads, head_dim]")
    if block_table.dim() != 2 or block_table.shape[0] != q.shape[0] or seq_lens.shape != (q.shape[0],):
        raise ValueError("block_table must be [S, max_blocks] and seq_lens [S]")
    if ring_k.shape != ring_v.shape or ring_k.dim() != 4 or ring_k.shape[0] != q.shape[0]:
        raise ValueError("ring_k and ring_v must be [S, R, H, d]")
    _token_rows(ring_k, "ring_k", cache.num_kv_heads, cfg.head_dim, ring=True)
    desc = cache.descriptor()
    _check(lib().tq_decode_attention_ring(
        ctypes.byref(cfg), _dev(q, torch.bfloat16, "q"), q.shape[0], q.shape[1], ctypes.byref(desc),
        _dev(block_table, torch.int32, "block_table"), block_table.shape[1],
        _dev(seq_lens, torch.int32, "seq_lens"), int(max_seq_len), float(sm_scale), int(num_splits),
        _dev(ring_k, torch.bfloat16, "ring_k"), _dev(ring_v, torch.bfloat16, "ring_v"), ring_k.shape[1],
        _dev(out, torch.float32, "out"), _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
        _stream(stream)))


def tq_dequant(cfg: TqConfig, cache: PagedCache, block_table: torch.Tensor, cu_seqlens: torch.Tensor,
               max_seq_len: int, k_out: torch.Tensor, v_out: torch.Tensor, stream=None):
    """k_out, v_out: bf16 [cu_seqlens[-1], H, d]; cu_seqlens int32 [S + 1].
    The row count of k_out and v_out is the caller's to get right (reading
    cu_seqlens[-1] here would synchronise the stream)."""
    if block_table.dim() != 2 or cu_seqlens.shape != (block_table.shape[0] + 1,):
        raise ValueError("block_table must be [S, max_blocks] and cu_seqlens [S + 1]")
    if v_out.shape != k_out.shape:
        raise ValueError("k_out and v_out must have the same shape")
    _token_rows(k_out, "k_out", cache.num_kv_heads, cfg.head_dim)
    desc = cache.descriptor()
    _check(lib().tq_dequant(
        ctypes.byref(cfg), ctypes.byref(desc), _dev(block_table, torch.int32, "block_table"),
        block_table.shape[1], _dev(cu_seqlens, torch.int32, "cu_seqlens"), block_table.shape[0],
        int(max_seq_len), _dev(k_out, torch.bfloat16, "k_out"), _dev(v_out, torch.bfloat16, "v_out"),
        _stream(stream)))
