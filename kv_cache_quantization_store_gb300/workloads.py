"""Seeded synthetic workloads for the TurboQuant store and decode path.

This module draws inputs only: keys, values, queries, sequence lengths,
block tables and slot mappings.  It holds none of the quantisation or
attention arithmetic, so the CPU oracle and the CUDA path can both be fed
from it.

All draws come from NumPy PCG64 generators keyed by ``(data_seed, stream,
chunk)``.  Any token range can therefore be regenerated on its own, and a
result does not depend on the thread count.  Floats are drawn in fp32 and
rounded once to bf16 (round to nearest even); the arrays returned here hold
those bf16 values as float32.

The five named workloads follow the configurations that TurboQuantConfig's
presets are measured on: the dataclass defaults at d=64, then k3v4_nc,
k8v4, 3bit_nc and 4bit_nc.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

#: tokens per generator chunk; chunk c of a workload uses rng (data_seed, STREAM_KV, c)
CHUNK_TOKENS = 4096
STREAM_KV = 1
STREAM_Q = 2
STREAM_OUTLIERS = 3
STREAM_LAYOUT = 4
STREAM_LENS = 5


def bf16_values(x: np.ndarray) -> np.ndarray:
    """fp32 array -> the nearest bf16 values (ties to even), as float32."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


@dataclass
class Workload:
    name: str
    head_dim: int
    key_bits: int
    value_bits: int
    norm_correction: bool
    num_kv_heads: int
    num_q_heads: int
    block_size: int
    seq_lens: np.ndarray
    data_seed: int
    kv_mode: str = "normal"          # "normal" | "outliers" | "lognormal"
    identity_blocks: bool = False
    layers: tuple = (0,)
    preset: str | None = None
    seed: int = 42
    block_stride: int | None = None  # bytes; None = dense blocks
    store_tokens: int | None = None  # bulk-store size of the timed step
    description: str = ""
    _layout: tuple | None = field(default=None, repr=False)

    # -- sizes ------------------------------------------------------------
    @property
    def num_seqs(self) -> int:
        return len(self.seq_lens)

    @property
    def num_tokens(self) -> int:
        return int(np.sum(self.seq_lens))

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def blocks_per_seq(self) -> np.ndarray:
        return (self.seq_lens + self.block_size - 1) // self.block_size

    # -- paged layout -----------------------------------------------------
    def layout(self):
        """(block_table int32 [S, max_blocks], num_blocks): every sequence
        gets exactly the blocks it needs, in a random order (identity order
        for workloads that ask for it); unused table entries are 0."""
        if self._layout is None:
            nblk = self.blocks_per_seq()
            total = int(nblk.sum())
            if self.identity_blocks:
                perm = np.arange(total)
            else:
                perm = np.random.default_rng([self.data_seed, STREAM_LAYOUT]).permutation(total)
            table = np.zeros((self.num_seqs, int(nblk.max()) if total else 1), dtype=np.int32)
            off = 0
            for s, n in enumerate(nblk):
                table[s, :n] = perm[off:off + n]
                off += n
            self._layout = (table, total)
        return self._layout

    def token_seq_pos(self):
        """For every cached token in order: (sequence id, position)."""
        seq = np.repeat(np.arange(self.num_seqs), self.seq_lens)
        starts = np.concatenate([[0], np.cumsum(self.seq_lens)[:-1]])
        pos = np.arange(self.num_tokens) - np.repeat(starts, self.seq_lens)
        return seq, pos

    def slot_mapping(self) -> np.ndarray:
        """int64 [T]: slot = block * block_size + offset for every cached token."""
        table, _ = self.layout()
        seq, pos = self.token_seq_pos()
        return (table[seq, pos // self.block_size].astype(np.int64) * self.block_size
                + pos % self.block_size)

    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.seq_lens)]).astype(np.int32)

    # -- tensors ----------------------------------------------------------
    def _outlier_channels(self):
        rng = np.random.default_rng([self.data_seed, STREAM_OUTLIERS])
        h, d = self.num_kv_heads, self.head_dim
        k_ch = np.stack([rng.choice(d, 4, replace=False) for _ in range(h)])
        v_ch = np.stack([rng.choice(d, 4, replace=False) for _ in range(h)])
        return k_ch, v_ch

    def _chunk(self, c: int):
        h, d = self.num_kv_heads, self.head_dim
        n = min(CHUNK_TOKENS, self.num_tokens - c * CHUNK_TOKENS)
        rng = np.random.default_rng([self.data_seed, STREAM_KV, c])
        k = rng.standard_normal((CHUNK_TOKENS, h, d), dtype=np.float32)[:n]
        v = rng.standard_normal((CHUNK_TOKENS, h, d), dtype=np.float32)[:n]
        if self.kv_mode == "outliers":
            k_ch, v_ch = self._outlier_channels()
            for hh in range(h):
                k[:, hh, k_ch[hh]] *= 10.0
                v[:, hh, v_ch[hh]] *= 10.0
        elif self.kv_mode == "lognormal":
            fk = np.exp(0.5 * rng.standard_normal(CHUNK_TOKENS)).astype(np.float32)[:n]
            fv = np.exp(0.5 * rng.standard_normal(CHUNK_TOKENS)).astype(np.float32)[:n]
            k *= fk[:, None, None]
            v *= fv[:, None, None]
        return bf16_values(k), bf16_values(v)

    def kv(self, start: int = 0, stop: int | None = None, threads: int | None = None):
        """Keys and values of cached tokens [start, stop): float32 [n, H, d] each."""
        stop = self.num_tokens if stop is None else stop
        h, d = self.num_kv_heads, self.head_dim
        k = np.empty((stop - start, h, d), dtype=np.float32)
        v = np.empty_like(k)
        chunks = range(start // CHUNK_TOKENS, (stop + CHUNK_TOKENS - 1) // CHUNK_TOKENS)

        def fill(c):
            kc, vc = self._chunk(c)
            lo = max(start, c * CHUNK_TOKENS)
            hi = min(stop, c * CHUNK_TOKENS + kc.shape[0])
            k[lo - start:hi - start] = kc[lo - c * CHUNK_TOKENS:hi - c * CHUNK_TOKENS]
            v[lo - start:hi - start] = vc[lo - c * CHUNK_TOKENS:hi - c * CHUNK_TOKENS]

        nthreads = threads or min(16, os.cpu_count() or 1)
        if len(chunks) > 1 and nthreads > 1:
            with ThreadPoolExecutor(nthreads) as ex:
                list(ex.map(fill, chunks))
        else:
            for c in chunks:
                fill(c)
        return k, v

    def kv_device(self, device, start: int = 0, stop: int | None = None):
        """Keys and values of tokens [start, stop) drawn on the device: bf16
        [n, H, d] each, with the workload's distribution (N(0,1), outlier
        channels x10 or a per-token LogNormal(0, 0.5) factor) from torch's
        generator seeded with (data_seed, STREAM_KV).  These are a second,
        faster source of the same distribution for timing runs; they are not
        the values ``kv`` returns."""
        stop = self.num_tokens if stop is None else stop
        n, h, d = stop - start, self.num_kv_heads, self.head_dim
        g = torch.Generator(device=device)
        g.manual_seed(self.data_seed * 1_000_003 + STREAM_KV * 7919 + start)
        out = []
        k_ch, v_ch = self._outlier_channels() if self.kv_mode == "outliers" else (None, None)
        for ch in (k_ch, v_ch):
            x = torch.randn((n, h, d), generator=g, device=device, dtype=torch.float32)
            if self.kv_mode == "outliers":
                for hh in range(h):
                    x[:, hh, torch.as_tensor(ch[hh], device=device)] *= 10.0
            elif self.kv_mode == "lognormal":
                x *= torch.exp(0.5 * torch.randn((n, 1, 1), generator=g, device=device, dtype=torch.float32))
            out.append(x.to(torch.bfloat16))
            del x
        return out[0], out[1]

    def q(self) -> np.ndarray:
        rng = np.random.default_rng([self.data_seed, STREAM_Q])
        x = rng.standard_normal((self.num_seqs, self.num_q_heads, self.head_dim), dtype=np.float32)
        return bf16_values(x)


def _lens(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    return np.random.default_rng([seed, STREAM_LENS]).integers(lo, hi + 1, size=n).astype(np.int64)


def named(name: str) -> Workload:
    """The five configurations, c0..c4, at full size."""
    if name == "c0":
        return Workload("c0", 64, 3, 4, False, 1, 2, 16, np.array([256]), 1000,
                        identity_blocks=True,
                        description="dataclass defaults (3-bit MSE keys, 4-bit values, no NC), "
                                    "d=64, 2 q / 1 kv head, 1 x 256 tokens, block 16")
    if name == "c1":
        return Workload("c1", 128, 3, 4, True, 8, 32, 16, _lens(1001, 8, 1024, 4096), 1001,
                        kv_mode="outliers", preset="turboquant_k3v4_nc",
                        description="turboquant_k3v4_nc d=128, 32 q / 8 kv heads, 8 seqs of "
                                    "U[1024,4096] tokens, 4 outlier channels x10 per head")
    if name == "c2":
        return Workload("c2", 128, 8, 4, False, 8, 32, 16, np.full(64, 8192), 1002,
                        kv_mode="lognormal", preset="turboquant_k8v4",
                        description="turboquant_k8v4 d=128, 32 q / 8 kv heads, 64 x 8192 tokens, "
                                    "per-token LogNormal(0,0.5) scale")
    if name == "c3":
        return Workload("c3", 128, 3, 3, True, 8, 40, 16, np.full(4, 131072), 1003,
                        kv_mode="outliers", preset="turboquant_3bit_nc",
                        description="turboquant_3bit_nc d=128, 40 q / 8 kv heads, 4 x 131072 "
                                    "tokens, 4 outlier channels x10 per head")
    if name == "c4":
        # lcm(tq page 4*262 B, bf16 skip page 2*4*256*2 B) = 536576 B per page,
        # which holds 512 TQ tokens: block_size 512, dense block stride.
        return Workload("c4", 256, 4, 4, True, 4, 16, 512, np.full(256, 2048), 1004,
                        layers=(0, 1, 2, 3), preset="turboquant_4bit_nc", store_tokens=65536,
                        description="turboquant_4bit_nc d=256, 16 q / 4 kv heads, 4 layers, "
                                    "lcm page (block 512), store 65536 tok + decode 256 x 2048")
    raise KeyError(name)


def small(name: str, seq_lens, **kw) -> Workload:
    """A configuration's format and head geometry on a small, ragged batch."""
    base = named(name)
    w = Workload(base.name + "-small", base.head_dim, base.key_bits, base.value_bits,
                 base.norm_correction, base.num_kv_heads, base.num_q_heads, base.block_size,
                 np.asarray(seq_lens, dtype=np.int64), base.data_seed + 100, kv_mode=base.kv_mode,
                 layers=base.layers, preset=base.preset)
    for key, val in kw.items():
        setattr(w, key, val)
    return w


def custom(head_dim: int, key_bits: int, value_bits: int, nc: bool, num_kv_heads: int,
           num_q_heads: int, block_size: int, seq_lens, data_seed: int, **kw) -> Workload:
    return Workload(f"d{head_dim}k{key_bits}v{value_bits}{'nc' if nc else ''}", head_dim, key_bits,
                    value_bits, nc, num_kv_heads, num_q_heads, block_size,
                    np.asarray(seq_lens, dtype=np.int64), data_seed, **kw)


def max_blocks(seq_len: int, block_size: int) -> int:
    return max(1, math.ceil(seq_len / block_size))
