"""Synthetic quality of the packed cache: relative MSE and cosine similarity
of the dequantised keys and values against the bf16 inputs, per preset, with
norm correction on and off.

[TQC] TurboQuantConfig docstring: the presets and the norm_correction line
(re-normalising the centroid vectors fixes the norm distortion).  [ART]
hnwysp.cn article, "Direction 2": per-preset accuracy trade-offs.  This is
context only: synthetic inputs with the five configurations' distributions,
no model and no perplexity.

It runs the product path on the GPU (tq_store_kv, then tq_dequant) and
measures with torch on the device:

    python -m kv_cache_quantization_store_gb300.quality [--tokens N] [--json]
"""
from __future__ import annotations

import argparse
import json

import numpy as np
import torch

import kv_cache_quantization_store_gb300 as tq
from kv_cache_quantization_store_gb300 import workloads as W

#: preset name -> (key bits, value bits, norm correction)  ([TQC] docstring presets)
PRESETS = {
    "turboquant_k8v4": (8, 4, False),
    "turboquant_4bit_nc": (4, 4, True),
    "turboquant_k3v4_nc": (3, 4, True),
    "turboquant_3bit_nc": (3, 3, True),
}
DISTRIBUTIONS = ("normal", "outliers", "lognormal")


def _metrics(x: torch.Tensor, y: torch.Tensor) -> tuple[float, float]:
    """(sum |x - y|^2 / sum |x|^2, mean cosine similarity) over the vectors."""
    x = x.float().reshape(-1, x.shape[-1])
    y = y.float().reshape(-1, y.shape[-1])
    rel = float(((x - y) ** 2).sum() / (x ** 2).sum())
    cos = float(torch.nn.functional.cosine_similarity(x, y, dim=1, eps=1e-30).mean())
    return rel, cos


def measure(key_bits: int, value_bits: int, head_dim: int, kv_mode: str, tokens: int, device,
            nc_options=(False, True)) -> list[dict]:
    """Stores `tokens` tokens of 8 KV heads once, dequantises them with norm
    correction off and on (the cache bytes do not depend on it), and returns
    one row per setting."""
    wl = W.custom(head_dim, key_bits, value_bits, False, 8, 32, 16, [tokens], 3000 + head_dim + key_bits,
                  kv_mode=kv_mode)
    k_np, v_np = wl.kv()
    k = torch.from_numpy(k_np).to(torch.bfloat16).to(device)
    v = torch.from_numpy(v_np).to(torch.bfloat16).to(device)
    table_np, nblk = wl.layout()
    table = torch.from_numpy(table_np).to(device)
    slots = torch.from_numpy(wl.slot_mapping()).to(device)
    cu = torch.from_numpy(wl.cu_seqlens()).to(device)
    rows = []
    cache = None
    for nc in (nc_options if key_bits != 8 else (False,)):
        cfg = tq.tq_config_init(head_dim, key_bits, value_bits, nc, wl.seed)
        if cache is None:
            cache = tq.new_paged_cache(cfg, nblk, wl.block_size, wl.num_kv_heads, 0, device=device)
            tq.tq_store_kv(cfg, k, v, slots, cache)
        k_hat = torch.empty_like(k)
        v_hat = torch.empty_like(v)
        tq.tq_dequant(cfg, cache, table, cu, tokens, k_hat, v_hat)
        torch.cuda.synchronize()
        if cache.error_flags():
            raise RuntimeError(f"cache error flags {cache.error_flags()}")
        k_rel, k_cos = _metrics(k, k_hat)
        v_rel, v_cos = _metrics(v, v_hat)
        rows.append({"key_bits": key_bits, "value_bits": value_bits, "norm_correction": nc, "kv": kv_mode,
                     "head_dim": head_dim, "tokens": tokens, "key_rel_mse": k_rel, "key_cos": k_cos,
                     "value_rel_mse": v_rel, "value_cos": v_cos,
                     "compression_vs_bf16": round(4 * head_dim / cfg.slot_size_aligned, 3)})
    return rows


def report(tokens: int = 16384, head_dim: int = 128, device=None) -> list[dict]:
    device = device or torch.device("cuda", 0)
    out = []
    for name, (kb, vb, _) in PRESETS.items():
        for mode in DISTRIBUTIONS:
            for row in measure(kb, vb, head_dim, mode, tokens, device):
                row["preset"] = name
                out.append(row)
    return out


def markdown(rows: list[dict]) -> str:
    lines = ["| preset | NC | K/V input | key rel. MSE | key cos | value rel. MSE | value cos | compression |",
             "|---|---|---|---:|---:|---:|---:|---:|"]
    for r in rows:
        lines.append(f"| {r['preset']} | {'on' if r['norm_correction'] else 'off'} | {r['kv']} | "
                     f"{r['key_rel_mse']:.5f} | {r['key_cos']:.5f} | {r['value_rel_mse']:.5f} | "
                     f"{r['value_cos']:.5f} | {r['compression_vs_bf16']}x |")
    return "\n".join(lines)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--tokens", type=int, default=16384)
    ap.add_argument("--head-dim", type=int, default=128)
    ap.add_argument("--json", action="store_true")
    args = ap.parse_args(argv)
    rows = report(args.tokens, args.head_dim)
    print(json.dumps(rows) if args.json else markdown(rows))


if __name__ == "__main__":
    main()
