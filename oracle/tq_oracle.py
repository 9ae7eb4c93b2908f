"""CPU oracle for the TurboQuant KV-cache store and fused decode attention.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, independent
statement of what the CUDA path must compute.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline legs of ``bench.py`` may
import it; the library (``kv_cache_quantization_store_gb300``) never does, and
it shares no code, table or constant generator with the CUDA sources.

Everything is NumPy.  Floating point is fp64, except the value quantiser,
whose integer codes are decided in IEEE fp32 exactly as stated in
``encode_values`` (the reading documented there), and the fp16 / fp32 / e4m3
roundings that the stored format itself fixes.

Sources (cited by page title and section):
  [TQC]  vLLM API docs, "vllm.model_executor.layers.quantization.turboquant",
         class TurboQuantConfig: docstring (presets, seed rule, norm
         correction), properties key_fp8 / mse_bits / key_packed_size /
         value_packed_size / slot_size / slot_size_aligned, from_cache_dtype.
  [PR]   prhub digest of vLLM PR #39931 "TurboQuant supports hybrid models +
         fixes page-size alignment", section "key source snippet"
         (vllm/platforms/interface.py, _align_hybrid_block_size).
  [ART]  hnwysp.cn TurboQuant article, section "Direction 1: fused Triton
         kernels" (rotate the query, online softmax block by block), and
         section "full_tq zero-allocation mode", item 3 (the write path: an
         exact bf16 ring of 128 tokens, compressed a whole block at a time).

Pins (tests/test_oracle_pins.py): slot sizes and the compression column of
the [TQC] preset table, the per-layer seed rule, published SplitMix64 test
vectors, Sylvester-Hadamard orthogonality and the FWHT, Lloyd-Max fixed-point
conditions plus Max's (1960) published N(0,1) quantiser tables and the 1-bit
closed form sqrt(2/pi), fp32 centroids and boundaries against an
independent 40-digit solve (boundaries: the correctly rounded exact
midpoint, not the midpoint of the fp32 centroids), exhaustive e4m3 encode
against a brute-force nearest search, value-quantiser invariants and
hand-worked rows that fix its readings (codes against the fp16 scale and
zero, ties to even), brute-force decode special cases,
split invariance of the log-sum-exp merge, and for the ring: token-by-token
appends equal one plain store of the whole blocks (bytes) with the rest
verbatim in the ring, chunked appends equal single steps, and the ring
decode reduces to the packed decode or to closed forms (one token, equal
keys).

Parity unpinned: byte-for-byte agreement with vLLM's own cache.  The pages do
not print the random-sign generator, the Hadamard row order or TQ_PRESETS, so
those are readings (listed where they are used), and only the agreement
between this oracle and the CUDA path is checked.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

# ---------------------------------------------------------------------------
# Configuration and sizes  ([TQC] TurboQuantConfig)
# ---------------------------------------------------------------------------

#: [TQC] docstring "Named presets": (key bits, value bits, norm correction).
#: TQ_PRESETS itself is not printed; this mapping is read off the preset
#: names and the docstring's one-line descriptions.
PRESETS = {
    "turboquant_k8v4": (8, 4, False),
    "turboquant_4bit_nc": (4, 4, True),
    "turboquant_k3v4_nc": (3, 4, True),
    "turboquant_3bit_nc": (3, 3, True),
}

#: [TQC] dataclass default seed.
DEFAULT_SEED = 42
#: [TQC] docstring "Actual seed per layer = seed + layer_idx * 1337".
LAYER_SEED_STRIDE = 1337


@dataclass(frozen=True)
class Config:
    """[TQC] TurboQuantConfig fields and derived sizes, restated."""

    head_dim: int = 128
    key_quant_bits: int = 3
    value_quant_bits: int = 4
    seed: int = DEFAULT_SEED
    norm_correction: bool = False

    @property
    def key_fp8(self) -> bool:
        # [TQC] key_fp8: 8 key bits means raw FP8 keys.
        return self.key_quant_bits == 8

    @property
    def mse_bits(self) -> int:
        # [TQC] mse_bits: FP8 mode still builds a value-width codebook.
        return self.value_quant_bits if self.key_fp8 else self.key_quant_bits

    @property
    def key_mse_bits(self) -> int:
        return 0 if self.key_fp8 else self.key_quant_bits

    @property
    def n_centroids(self) -> int:
        return 1 << self.mse_bits

    @property
    def key_packed_size(self) -> int:
        # [TQC] key_packed_size: d bytes for FP8, else index bytes + fp16 norm.
        if self.key_fp8:
            return self.head_dim
        return _ceil_div(self.head_dim * self.key_mse_bits, 8) + 2

    @property
    def value_packed_size(self) -> int:
        # [TQC] value_packed_size: code bytes + fp16 scale + fp16 zero.
        return _ceil_div(self.head_dim * self.value_quant_bits, 8) + 4

    @property
    def slot_size(self) -> int:
        return self.key_packed_size + self.value_packed_size

    @property
    def slot_size_aligned(self) -> int:
        # [TQC] slot_size_aligned: next even number.
        s = self.slot_size
        return s + (s & 1)


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def config_from_preset(name: str, head_dim: int) -> Config:
    """[TQC] from_cache_dtype: unknown names raise ValueError naming the valid ones."""
    if name not in PRESETS:
        raise ValueError(f"unknown TurboQuant preset {name!r}; valid: {', '.join(PRESETS)}")
    kb, vb, nc = PRESETS[name]
    return Config(head_dim=head_dim, key_quant_bits=kb, value_quant_bits=vb, norm_correction=nc)


def layer_seed(seed: int, layer_idx: int) -> int:
    """[TQC] docstring, Args/seed: per-layer seed rule."""
    return seed + layer_idx * LAYER_SEED_STRIDE


# ---------------------------------------------------------------------------
# Paged-cache geometry  ([PR] interface.py snippet)
# ---------------------------------------------------------------------------

def tq_page_bytes_per_token(num_kv_heads: int, slot_size_aligned: int) -> int:
    """Bytes one token occupies in a TQ layer: every KV head's packed slot.

    Reading of [PR]'s TQFullAttentionSpec(block_size=1, ..., tq_slot_size=...)
    page size: heads x slot bytes (the spec's formula is not printed).
    """
    return num_kv_heads * slot_size_aligned


def skip_page_bytes_per_token(num_kv_heads: int, head_dim: int, dtype_bytes: int = 2) -> int:
    """Bytes one token occupies in an unquantised (skip) layer: K and V.

    Reading of [PR]'s FullAttentionSpec(block_size=1, ...) page size:
    2 (K and V) x heads x head_dim x dtype bytes.
    """
    return 2 * num_kv_heads * head_dim * dtype_bytes


def hybrid_page_bytes(tq_page: int, skip_page: int | None) -> int:
    """[PR] snippet: with skip layers present the per-token page is lcm(tq, skip)."""
    if not skip_page:
        return tq_page
    return tq_page * skip_page // math.gcd(tq_page, skip_page)


# ---------------------------------------------------------------------------
# Random signs and the rotation
# ---------------------------------------------------------------------------

_MASK64 = (1 << 64) - 1


def splitmix64(seed: int, n: int) -> list[int]:
    """SplitMix64 (Steele, Lea & Flood, OOPSLA 2014): n successive outputs.

    State advances by the golden-gamma constant; each output is the state
    passed through the published 64-bit finaliser (xor-shift 30, multiply,
    xor-shift 27, multiply, xor-shift 31).
    """
    state = seed & _MASK64
    out = []
    for _ in range(n):
        state = (state + 0x9E3779B97F4A7C15) & _MASK64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
        out.append(z ^ (z >> 31))
    return out


def random_signs(seed_l: int, d: int) -> np.ndarray:
    """Diagonal of the random-sign matrix for one layer.

    [TQC] only says "deterministic random matrix generation" from the layer
    seed.  Reading: draw i of a SplitMix64 stream seeded with the layer seed
    gives s_i = -1 when its top bit is set, else +1.
    """
    return np.array([-1.0 if (x >> 63) else 1.0 for x in splitmix64(seed_l, d)])


def sylvester_hadamard(d: int) -> np.ndarray:
    """Natural-order Sylvester Hadamard matrix: H_1 = [1], H_2m = [[H, H], [H, -H]]."""
    if d < 1 or d & (d - 1):
        raise ValueError("Hadamard order must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def rotation_matrix(signs: np.ndarray) -> np.ndarray:
    """Pi = H_d diag(s) / sqrt(d): the random-sign Walsh-Hadamard rotation.

    [TQC] docstring names the key transform "WHT rotation"; the ordering
    (signs first, then Hadamard) is a reading.
    """
    d = signs.shape[0]
    return sylvester_hadamard(d) * signs[None, :] / math.sqrt(d)


# ---------------------------------------------------------------------------
# Lloyd-Max scalar quantiser for N(0, 1/d)
# ---------------------------------------------------------------------------

def _phi(x: float) -> float:
    return 0.0 if math.isinf(x) else math.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)


def _Phi(x: float) -> float:
    return 0.5 * math.erfc(-x / math.sqrt(2.0))


def lloyd_max_normal(levels: int, tol: float = 1e-13, max_iter: int = 100_000):
    """Lloyd-Max quantiser of the standard normal, by fixed-point iteration.

    Start from the uniform grid on [-3, 3]; alternately put each boundary at
    the midpoint of its neighbouring centroids and each centroid at the mean
    of N(0,1) over its cell, (phi(a) - phi(b)) / (Phi(b) - Phi(a)); keep the
    grid symmetric about 0; stop once no centroid moves by ``tol``.
    Returns (centroids, iterations) in fp64.
    """
    c = np.linspace(-3.0, 3.0, levels)
    for it in range(1, max_iter + 1):
        b = 0.5 * (c[:-1] + c[1:])
        edges = [-math.inf] + list(b) + [math.inf]
        new = np.array([
            (_phi(edges[j]) - _phi(edges[j + 1])) / (_Phi(edges[j + 1]) - _Phi(edges[j]))
            for j in range(levels)
        ])
        new = 0.5 * (new - new[::-1])
        moved = float(np.max(np.abs(new - c)))
        c = new
        if moved < tol:
            return c, it
    raise RuntimeError("Lloyd-Max iteration did not converge")


@dataclass(frozen=True)
class Codebook:
    centroids: np.ndarray   # fp32 values (held as float32), ascending
    boundaries: np.ndarray  # fp32 decision thresholds, ascending, len = levels - 1
    sigma: float


def codebook(head_dim: int, bits: int) -> Codebook:
    """Centroids and boundaries for the rotated coordinate, N(0, 1/d).

    A unit vector after a random rotation has coordinates close to N(0, 1/d);
    the N(0,1) quantiser is scaled by sigma = 1/sqrt(d), rounded to fp32, and
    each fp32 boundary is the fp64 midpoint of its two scaled centroids
    rounded to fp32.
    """
    sigma = 1.0 / math.sqrt(head_dim)
    c, _ = lloyd_max_normal(1 << bits)
    cs = c * sigma
    return Codebook(
        centroids=cs.astype(np.float32),
        boundaries=(0.5 * (cs[:-1] + cs[1:])).astype(np.float32),
        sigma=sigma,
    )


# ---------------------------------------------------------------------------
# Bit packing, fp16 / bf16 / e4m3 codecs
# ---------------------------------------------------------------------------

def pack_bits(codes: np.ndarray, bits: int) -> np.ndarray:
    """LSB-first bitstream: code i fills bits [i*bits, (i+1)*bits) of the bytes.

    codes: [N, n] non-negative ints below 2**bits -> uint8 [N, ceil(n*bits/8)].
    Eight consecutive codes fill exactly ``bits`` bytes: their integer
    sum(code_j << (bits * j)) written little-endian.
    """
    codes = np.asarray(codes, dtype=np.int64)
    n_vec, n = codes.shape
    groups = -(-n // 8)
    padded = np.zeros((n_vec, groups * 8), dtype=np.int64)
    padded[:, :n] = codes
    word = np.zeros((n_vec, groups), dtype=np.int64)
    for j in range(8):
        word |= padded[:, j::8] << (bits * j)
    out = np.stack([(word >> (8 * m)) & 0xFF for m in range(bits)], axis=2).astype(np.uint8)
    return out.reshape(n_vec, groups * bits)[:, : -(-n * bits // 8)]


def unpack_bits(data: np.ndarray, bits: int, n: int) -> np.ndarray:
    """Inverse of pack_bits: uint8 [N, nbytes] -> int64 [N, n]."""
    data = np.asarray(data, dtype=np.uint8)
    n_vec = data.shape[0]
    groups = -(-n // 8)
    full = np.zeros((n_vec, groups * bits), dtype=np.int64)
    full[:, : data.shape[1]] = data[:, : groups * bits]
    full = full.reshape(n_vec, groups, bits)
    word = np.zeros((n_vec, groups), dtype=np.int64)
    for m in range(bits):
        word |= full[:, :, m] << (8 * m)
    out = np.stack([(word >> (bits * j)) & ((1 << bits) - 1) for j in range(8)], axis=2)
    return out.reshape(n_vec, groups * 8)[:, :n]


def f16_bytes(x: np.ndarray) -> np.ndarray:
    """fp16 values -> little-endian byte pairs [N, 2]."""
    return np.ascontiguousarray(np.asarray(x, dtype="<f2")).view(np.uint8).reshape(-1, 2)


def f16_from_bytes(b: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(b, dtype=np.uint8).view("<f2").reshape(-1).astype(np.float64)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns float32 values."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    is_nan = np.isnan(np.asarray(x, dtype=np.float32))
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    r = np.where(is_nan, (u >> 16) | 0x40, r).astype(np.uint32)
    return (r << 16).astype(np.uint32).view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Bit patterns (uint16) of bf16 values held exactly in float32."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


E4M3_MAX = 448.0


def e4m3_value(code: int) -> float:
    """Real value of an OCP FP8 E4M3 (fn) byte; NaN for S.1111.111."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return s * m * 2.0 ** -9
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """OCP FP8 E4M3 encode, round to nearest even, saturating to +-448.

    [TQC] key_fp8 stores one byte per element; the rounding and saturation
    rules are not printed, so this is a reading (saturation never triggers at
    the configured input scales).  Exponent bias 7, 3 mantissa bits,
    subnormal quantum 2**-9.  NaN inputs map to 0x7F.
    """
    x = np.asarray(x, dtype=np.float64).reshape(-1)
    out = np.empty(x.shape, dtype=np.uint8)
    for i, v in enumerate(x):
        if math.isnan(v):
            out[i] = 0x7F
            continue
        sign = 0x80 if math.copysign(1.0, v) < 0 else 0
        a = min(abs(v), E4M3_MAX) if math.isfinite(v) else E4M3_MAX
        if a < 2.0 ** -6:
            quantum = 2.0 ** -9
        else:
            quantum = 2.0 ** (math.floor(math.log2(a)) - 3)
        q = round(a / quantum) * quantum  # Python round(): ties to even
        q = min(q, E4M3_MAX)
        if q == 0.0:
            out[i] = sign
        elif q < 2.0 ** -6:
            out[i] = sign | int(q / 2.0 ** -9)
        else:
            e = math.floor(math.log2(q))
            m = int(round((q / 2.0 ** e - 1.0) * 8))
            out[i] = sign | ((e + 7) << 3) | m
    return out


# ---------------------------------------------------------------------------
# Store path
# ---------------------------------------------------------------------------

def boundary_window(boundaries: np.ndarray, sigma: float) -> np.ndarray:
    """Half-width of the near-boundary window in which a key index is exempt
    from bit-exact parity: 1e-5 relative, with a floor of 1e-5*sigma so that
    the boundary at 0 has a window too (reading)."""
    b = np.asarray(boundaries, dtype=np.float64)
    return 1e-5 * np.maximum(np.abs(b), sigma)


def encode_keys_mse(k: np.ndarray, pi: np.ndarray, cb: Codebook):
    """Key MSE encode ([TQC] docstring "PolarQuant: WHT rotation + Lloyd-Max").

    k: [N, d] key vectors (bf16 values).  For each: n = ||k||_2; y = Pi k / n;
    idx_i = number of boundaries strictly below y_i; vec_norm = fp16(n).
    A zero key has y = 0 (so every index is the lower middle cell) and norm 0.
    Returns (idx [N, d] int64, vec_norm float16 [N], near [N, d] bool) where
    ``near`` marks coordinates inside the exemption window of a boundary.
    """
    k = np.asarray(k, dtype=np.float64)
    n = np.sqrt(np.sum(k * k, axis=1))
    safe = np.where(n > 0, n, 1.0)
    y = (k / safe[:, None]) @ pi.T
    y[n == 0] = 0.0
    b = cb.boundaries.astype(np.float64)
    # number of boundaries strictly below y
    idx = np.searchsorted(b, y, side="left")
    # the closest boundaries are the ones on either side of y
    win = boundary_window(b, cb.sigma)
    below = np.clip(idx - 1, 0, len(b) - 1)
    above = np.clip(idx, 0, len(b) - 1)
    near = (np.abs(y - b[below]) <= win[below]) | (np.abs(y - b[above]) <= win[above])
    return idx.astype(np.int64), n.astype(np.float16), near


def encode_values(v: np.ndarray, bits: int):
    """Uniform value quantiser ([TQC] value_packed_size: codes + fp16 scale + fp16 zero).

    Reading (the pages print sizes, not the formula), every step one IEEE fp32
    operation in this order: mn = min v, mx = max v; scale = fp16(fp32(mx - mn)
    / (2**bits - 1)); zero = fp16(mn); code_i = clamp(rint(fp32(v_i - zero) /
    scale), 0, 2**bits - 1) with the fp16-rounded scale and zero (the ones a
    reader sees), rint rounding half to even; a zero scale gives all-zero codes.
    v: [N, d] (bf16 values).  Returns (codes int64 [N, d], scale f16 [N], zero f16 [N]).
    """
    v = np.asarray(v, dtype=np.float32)
    top = np.float32((1 << bits) - 1)
    mn = v.min(axis=1)
    mx = v.max(axis=1)
    with np.errstate(over="ignore"):
        scale = ((mx - mn).astype(np.float32) / top).astype(np.float32).astype(np.float16)
        zero = mn.astype(np.float16)
    s32 = scale.astype(np.float32)
    z32 = zero.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        q = (v - z32[:, None]).astype(np.float32) / s32[:, None]
    codes = np.clip(np.rint(q), 0, top)
    codes = np.where(s32[:, None] == 0, 0, codes)
    return codes.astype(np.int64), scale, zero


@dataclass
class Layer:
    """A layer's key transform: config, codebook, signs and rotation."""

    cfg: Config
    layer_idx: int
    cb: Codebook
    signs: np.ndarray
    pi: np.ndarray


def make_layer(cfg: Config, layer_idx: int) -> Layer:
    signs = random_signs(layer_seed(cfg.seed, layer_idx), cfg.head_dim)
    return Layer(cfg, layer_idx, codebook(cfg.head_dim, cfg.mse_bits), signs, rotation_matrix(signs))


def encode_slots(layer: Layer, k: np.ndarray, v: np.ndarray):
    """Pack key/value vectors into slots [key_packed | value_packed | pad].

    [TQC] slot_size docstring gives the order; key_packed is [indices |
    vec_norm] (or d FP8 bytes), value_packed is [codes | scale | zero], fp16
    little-endian, pad byte 0.  k, v: [N, d].  Returns (slots uint8 [N,
    slot_size_aligned], near bool [N, d]) -- ``near`` flags key indices exempt
    from bit-exact parity (all False for FP8 keys).
    """
    cfg = layer.cfg
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n_vec, d = k.shape
    out = np.zeros((n_vec, cfg.slot_size_aligned), dtype=np.uint8)
    if cfg.key_fp8:
        out[:, :d] = e4m3_encode(k).reshape(n_vec, d)
        near = np.zeros((n_vec, d), dtype=bool)
    else:
        idx, vec_norm, near = encode_keys_mse(k, layer.pi, layer.cb)
        nb = cfg.key_packed_size - 2
        out[:, :nb] = pack_bits(idx, cfg.key_mse_bits)
        out[:, nb:nb + 2] = f16_bytes(vec_norm)
    codes, scale, zero = encode_values(v, cfg.value_quant_bits)
    o = cfg.key_packed_size
    nb = cfg.value_packed_size - 4
    out[:, o:o + nb] = pack_bits(codes, cfg.value_quant_bits)
    out[:, o + nb:o + nb + 2] = f16_bytes(scale)
    out[:, o + nb + 2:o + nb + 4] = f16_bytes(zero)
    return out, near


@dataclass
class PagedCache:
    """Paged byte cache [num_blocks, block_size, num_kv_heads, slot_size_aligned]
    with a block stride of ``block_stride`` bytes (>= the dense block size)."""

    data: np.ndarray  # uint8, flat, num_blocks * block_stride bytes
    num_blocks: int
    block_size: int
    num_kv_heads: int
    slot_bytes: int
    block_stride: int

    def slot_offset(self, slot: int, head: int) -> int:
        blk, pos = divmod(int(slot), self.block_size)
        return blk * self.block_stride + (pos * self.num_kv_heads + head) * self.slot_bytes


def new_cache(cfg: Config, num_blocks: int, block_size: int, num_kv_heads: int,
              block_stride: int | None = None) -> PagedCache:
    dense = block_size * num_kv_heads * cfg.slot_size_aligned
    stride = dense if block_stride is None else block_stride
    if stride < dense:
        raise ValueError("block stride smaller than a block")
    return PagedCache(np.zeros(num_blocks * stride, dtype=np.uint8), num_blocks, block_size,
                      num_kv_heads, cfg.slot_size_aligned, stride)


def store_kv(layer: Layer, k: np.ndarray, v: np.ndarray, slot_mapping: np.ndarray, cache: PagedCache):
    """Write tokens' packed slots into the paged cache.

    k, v: [T, H, d]; slot_mapping: [T] int, slot = block * block_size +
    position; a negative slot marks a padding token and is skipped (vLLM's
    convention; the pages do not print the store kernel).  Returns the
    exemption mask near [T, H, d].
    """
    t_n, h_n, d = k.shape
    slots, near = encode_slots(layer, k.reshape(-1, d), v.reshape(-1, d))
    slots = slots.reshape(t_n, h_n, -1)
    sm = np.asarray(slot_mapping, dtype=np.int64)
    keep = sm >= 0
    off = slot_offsets(cache, sm[keep])
    cache.data[off[..., None] + np.arange(cache.slot_bytes)] = slots[keep]
    return near.reshape(t_n, h_n, d)


def slot_offsets(cache: PagedCache, slots: np.ndarray) -> np.ndarray:
    """Byte offsets [T, H] of every KV head's slot for the given slot ids."""
    blk, pos = np.divmod(np.asarray(slots, dtype=np.int64), cache.block_size)
    heads = np.arange(cache.num_kv_heads)
    return (blk * cache.block_stride)[:, None] + (pos[:, None] * cache.num_kv_heads + heads[None, :]) * cache.slot_bytes


def read_slots(cache: PagedCache, block_table_row: np.ndarray, seq_len: int, head: int) -> np.ndarray:
    """Bytes of one KV head's slots for positions 0..seq_len-1 of a sequence."""
    pos = np.arange(seq_len)
    slots = np.asarray(block_table_row, dtype=np.int64)[pos // cache.block_size] * cache.block_size + pos % cache.block_size
    off = slot_offsets(cache, slots)[:, head]
    return cache.data[off[:, None] + np.arange(cache.slot_bytes)]


# ---------------------------------------------------------------------------
# Dequantisation
# ---------------------------------------------------------------------------

def dequant_slots(layer: Layer, slots: np.ndarray):
    """Packed slots [N, slot] -> (k_hat, v_hat) fp64 [N, d].

    Keys: k_hat = vec_norm * Pi^T c~, with c~ the centroid vector of the
    indices, divided by ||c~|| under norm correction ([TQC] docstring
    "norm_correction": centroid vectors renormalised to unit norm before the
    inverse rotation); FP8 keys decode the e4m3 bytes.
    Values: v_hat = scale * code + zero from the fp16 fields.
    """
    cfg = layer.cfg
    slots = np.asarray(slots, dtype=np.uint8)
    d = cfg.head_dim
    if cfg.key_fp8:
        table = np.array([e4m3_value(c) for c in range(256)])
        k_hat = table[slots[:, :d]]
    else:
        nb = cfg.key_packed_size - 2
        idx = unpack_bits(slots[:, :nb], cfg.key_mse_bits, d)
        norm = f16_from_bytes(slots[:, nb:nb + 2])
        c = layer.cb.centroids.astype(np.float64)[idx]
        if cfg.norm_correction:
            cn = np.sqrt(np.sum(c * c, axis=1))
            c = c / np.where(cn > 0, cn, 1.0)[:, None]
        k_hat = norm[:, None] * (c @ layer.pi)
    o = cfg.key_packed_size
    nb = cfg.value_packed_size - 4
    codes = unpack_bits(slots[:, o:o + nb], cfg.value_quant_bits, d)
    scale = f16_from_bytes(slots[:, o + nb:o + nb + 2])
    zero = f16_from_bytes(slots[:, o + nb + 2:o + nb + 4])
    v_hat = scale[:, None] * codes + zero[:, None]
    return k_hat, v_hat


def dequant_values_f32(layer: Layer, slots: np.ndarray) -> np.ndarray:
    """Values reconstructed in fp32 as fp32(scale) * code + fp32(zero) (the
    product is exact, so the sum is the one rounding), for the bf16 output of
    the continuation-prefill dequant."""
    cfg = layer.cfg
    o = cfg.key_packed_size
    nb = cfg.value_packed_size - 4
    codes = unpack_bits(slots[:, o:o + nb], cfg.value_quant_bits, cfg.head_dim).astype(np.float32)
    scale = f16_from_bytes(slots[:, o + nb:o + nb + 2]).astype(np.float32)
    zero = f16_from_bytes(slots[:, o + nb + 2:o + nb + 4]).astype(np.float32)
    return (scale[:, None] * codes + zero[:, None]).astype(np.float32)


def dequant_cache(layer: Layer, cache: PagedCache, block_table: np.ndarray, cu_seqlens: np.ndarray):
    """Continuation-prefill dequant ([TQC] mse_bits docstring): every cached
    token of every sequence back to bf16 K and V in varlen layout.

    Token j of sequence s lands in row cu_seqlens[s] + j.  Returns
    (k [rows, H, d], v [rows, H, d]) as bf16 values held in float32: keys
    rounded from fp64 to fp32 and then to bf16, values from the fp32
    reconstruction.
    """
    cfg = layer.cfg
    rows = int(cu_seqlens[-1])
    h_n = cache.num_kv_heads
    k_out = np.zeros((rows, h_n, cfg.head_dim), dtype=np.float32)
    v_out = np.zeros((rows, h_n, cfg.head_dim), dtype=np.float32)
    for s in range(len(cu_seqlens) - 1):
        start, n = int(cu_seqlens[s]), int(cu_seqlens[s + 1] - cu_seqlens[s])
        for h in range(h_n):
            sl = read_slots(cache, block_table[s], n, h)
            k_hat, _ = dequant_slots(layer, sl)
            k_out[start:start + n, h] = bf16_round(k_hat.astype(np.float32))
            v_out[start:start + n, h] = bf16_round(dequant_values_f32(layer, sl))
    return k_out, v_out


# ---------------------------------------------------------------------------
# Decode attention (brute force)
# ---------------------------------------------------------------------------

def attention_row(q: np.ndarray, k_hat: np.ndarray, v_hat: np.ndarray, sm_scale: float) -> np.ndarray:
    """softmax(sm_scale * K q) V for one query, fp64; an empty history gives 0."""
    if k_hat.shape[0] == 0:
        return np.zeros(v_hat.shape[1])
    s = (k_hat @ np.asarray(q, dtype=np.float64)) * sm_scale
    p = np.exp(s - s.max())
    return (p @ v_hat) / p.sum()


def decode_attention(layer: Layer, q: np.ndarray, cache: PagedCache, block_table: np.ndarray,
                     seq_lens: np.ndarray, sm_scale: float | None = None, rows=None) -> np.ndarray:
    """One decode step: every query head attends over its sequence's cache.

    q: [S, Hq, d].  Query head hq reads KV head hq // (Hq / H) (grouped-query
    convention; the pages are silent).  seq_lens counts the cached tokens
    attended to.  Scores use k_hat from ``dequant_slots`` -- the plain
    definition q . k_hat, where the fused kernel instead rotates q ([ART]
    "Direction 1"); both are the same number.  ``rows`` optionally limits the
    work to a list of (s, hq) pairs; other rows are left 0.
    Returns fp64 [S, Hq, d].
    """
    cfg = layer.cfg
    n_seq, hq_n, d = q.shape
    h_n = cache.num_kv_heads
    if hq_n % h_n:
        raise ValueError("query heads must be a multiple of KV heads")
    group = hq_n // h_n
    scale = 1.0 / math.sqrt(d) if sm_scale is None or sm_scale <= 0 else sm_scale
    out = np.zeros((n_seq, hq_n, d))
    wanted = None if rows is None else {}
    if rows is not None:
        for s, hq in rows:
            wanted.setdefault((s, hq // group), []).append(hq)
    for s in range(n_seq):
        for h in range(h_n):
            heads = range(h * group, (h + 1) * group) if wanted is None else wanted.get((s, h), [])
            if not heads:
                continue
            sl = read_slots(cache, block_table[s], int(seq_lens[s]), h)
            k_hat, v_hat = dequant_slots(layer, sl)
            for hq in heads:
                out[s, hq] = attention_row(q[s, hq], k_hat, v_hat, scale)
    return out


def partial_state(q: np.ndarray, k_hat: np.ndarray, v_hat: np.ndarray, sm_scale: float):
    """Split-KV partial for one query over a token range: (m, l, o~) with
    m = max score, l = sum exp(s - m), o~ = sum exp(s - m) v."""
    s = (k_hat @ np.asarray(q, dtype=np.float64)) * sm_scale
    m = s.max()
    p = np.exp(s - m)
    return m, p.sum(), p @ v_hat


def merge_partials(parts):
    """Log-sum-exp merge of split partials into the attention output."""
    m = max(p[0] for p in parts)
    lsum = sum(p[1] * math.exp(p[0] - m) for p in parts)
    o = sum(p[2] * math.exp(p[0] - m) for p in parts)
    return o / lsum


# ---------------------------------------------------------------------------
# Ring-buffered store  ([ART] hnwysp.cn article, "full_tq zero-allocation
# mode", item 3 "the write path": new decode tokens first go into an exact
# bf16 ring of 128 tokens, and only a full ring is compressed, a whole block
# at a time, so that no single token pays the quantiser on the hot path)
# ---------------------------------------------------------------------------

#: ring length the article names
RING_TOKENS = 128


def ring_split(seq_len: int, ring_tokens: int) -> tuple[int, int]:
    """(packed, in ring) token counts of a sequence of seq_len tokens.

    Reading (the article gives the ring's size and flush rule, not its
    alignment): ring blocks are aligned to multiples of the ring length from
    position 0, so the whole blocks are packed and the remainder waits in the
    ring, token p in ring row p mod R.
    """
    packed = (seq_len // ring_tokens) * ring_tokens
    return packed, seq_len - packed


def ring_append(layer: Layer, cache: PagedCache, block_table: np.ndarray, ring_k: np.ndarray, ring_v: np.ndarray,
                seq_lens: np.ndarray, k_new: np.ndarray, v_new: np.ndarray, cu_new: np.ndarray):
    """Append new tokens to sequences whose newest tokens wait in a ring.

    ring_k, ring_v: [S, R, H, d] exact rows, updated in place; seq_lens[s]:
    tokens of sequence s before the call (negative: the sequence takes no
    tokens); its new tokens are rows cu_new[s] .. cu_new[s+1]-1 of k_new,
    v_new [T, H, d], at positions seq_lens[s], seq_lens[s] + 1, ...  Every
    ring block that the new tokens complete is quantised into the packed
    cache at its positions (block_table gives the blocks); the tokens of the
    block that stays incomplete are written exactly into the ring.  A decode
    step is one new token per sequence.  Returns {(s, position): near mask
    [H, d]} for the tokens quantised by this call.
    """
    r_len = ring_k.shape[1]
    near_out = {}
    for s in range(len(seq_lens)):
        old = int(seq_lens[s])
        if old < 0:
            continue
        a, b = int(cu_new[s]), int(cu_new[s + 1])
        total = old + (b - a)
        old_packed, _ = ring_split(old, r_len)
        new_packed, _ = ring_split(total, r_len)
        # exact rows of positions old_packed .. total - 1: the ring's, then the new ones
        pos = np.arange(old_packed, total)
        rows_k = np.concatenate([ring_k[s, pos[pos < old] % r_len], k_new[a:b]])
        rows_v = np.concatenate([ring_v[s, pos[pos < old] % r_len], v_new[a:b]])
        full = pos < new_packed
        if full.any():
            p = pos[full]
            slots = np.asarray(block_table[s], dtype=np.int64)[p // cache.block_size] * cache.block_size \
                + p % cache.block_size
            near = store_kv(layer, rows_k[full], rows_v[full], slots, cache)
            for i, pp in enumerate(p):
                near_out[(s, int(pp))] = near[i]
        tail = ~full
        ring_k[s, pos[tail] % r_len] = rows_k[tail]
        ring_v[s, pos[tail] % r_len] = rows_v[tail]
    return near_out


def decode_attention_ring(layer: Layer, q: np.ndarray, cache: PagedCache, block_table: np.ndarray,
                          seq_lens: np.ndarray, ring_k: np.ndarray, ring_v: np.ndarray,
                          sm_scale: float | None = None) -> np.ndarray:
    """Decode over a packed history plus its exact ring (the article's
    hybrid mode: history from the compressed store, the newest tokens from
    the exact ring).  Sequence s of seq_lens[s] tokens attends over k_hat,
    v_hat of its ring_split packed tokens followed by the exact ring rows
    0 .. n - 1 (positions packed .. seq_len - 1).  Returns fp64 [S, Hq, d]."""
    cfg = layer.cfg
    n_seq, hq_n, d = q.shape
    h_n = cache.num_kv_heads
    group = hq_n // h_n
    r_len = ring_k.shape[1]
    scale = 1.0 / math.sqrt(d) if sm_scale is None or sm_scale <= 0 else sm_scale
    out = np.zeros((n_seq, hq_n, d))
    for s in range(n_seq):
        packed, n_ring = ring_split(max(int(seq_lens[s]), 0), r_len)
        for h in range(h_n):
            k_hat, v_hat = dequant_slots(layer, read_slots(cache, block_table[s], packed, h))
            k_all = np.concatenate([k_hat, ring_k[s, :n_ring, h].astype(np.float64)])
            v_all = np.concatenate([v_hat, ring_v[s, :n_ring, h].astype(np.float64)])
            for hq in range(h * group, (h + 1) * group):
                out[s, hq] = attention_row(q[s, hq], k_all, v_all, scale)
    return out
