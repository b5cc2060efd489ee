"""Seeded synthetic workloads shaped like the pages' configurations.

This module only draws random inputs (and builds the batch geometry that
describes them); it holds none of the method's arithmetic.  Tests feed the
same tensors to the CUDA path and, copied to the host, to the CPU oracle; the
bench uses them as its timed inputs.

Distributions: q, k, latent, K, V ~ N(0, 1) rounded to the storage dtype;
indexer weights w ~ N(0, 1/H) (config 1: U(0, 1)).  Seed = 1000 + config
number.  No dataset or trained weight is involved.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, Optional

import torch

CONFIGS = {
    1: "tiny prefill fp32: 1 seq x 256 tokens causal, indexer 4x32, top_k 64, MQA 4q/1kv d32",
    2: "decode: 8 seqs x n_kv 8192, bf16 q / F16 indexer cache 64x128, top_k 2048, MLA 128 heads 576/512",
    3: "prefill: 1 seq x 16384 tokens causal bf16, indexer 64x128 + Hadamard, top_k 2048, MLA 128 heads",
    4: "block-pooled decode: 16 seqs x 32768 bf16, C=64, indexer 32x128, top_k 2048, GQA 32q/4kv d128",
    5: "long-context decode: 64 seqs, n_kv ~ U[4096, 131072], F16 cache 64x128, top_k 2048, MLA 128 heads",
    "headline": "decode: 64 seqs x n_kv 131072, F16 indexer cache 64x128, top_k 2048, MLA 128 heads 576/512",
}


@dataclass
class Workload:
    name: str
    kind: str                      # "decode" | "prefill" | "block_decode"
    B: int
    T: int
    n_kv: torch.Tensor             # int32 [B] on device
    n_kv_host: list
    max_n_kv: int
    top_k: int
    H: int                         # indexer heads
    d: int                         # indexer head dim
    q_idx: torch.Tensor            # [B*T, H, d]
    w: torch.Tensor                # f32 [B*T, H]
    k_idx: torch.Tensor            # [rows, d] indexer keys (raw keys for block mode)
    scale: float
    q_attn: torch.Tensor           # [B*T, Hq, dk]
    k_attn: torch.Tensor           # MLA latent [rows, 576] or GQA K [rows, Hkv, dk]
    v_attn: Optional[torch.Tensor]  # GQA V [rows, Hkv, dv] or None (MLA)
    dv: int
    kv_start: Optional[torch.Tensor] = None
    kv_start_host: Optional[list] = None
    kv_seq_stride: int = 0
    q_pos: Optional[torch.Tensor] = None
    hadamard: bool = False
    block_size: int = 0
    page_table: Optional[torch.Tensor] = None   # int32 [B, pages]: paged caches (rows of page_size)
    page_size: int = 0
    k8: Optional[torch.Tensor] = None        # int8 indexer key codes [rows, >= d] (quantized cache)
    k_scale: Optional[torch.Tensor] = None   # f32 [rows] per-row scales of k8 (None: inline in the rows)
    extra: Dict = field(default_factory=dict)

    def row0(self, b: int) -> int:
        return self.kv_start_host[b] if self.kv_start_host is not None else b * self.kv_seq_stride

    def rows_of(self, b: int, n: int) -> torch.Tensor:
        """Cache rows of positions 0..n-1 of sequence b (through the page table if paged)."""
        j = torch.arange(n)
        if self.page_table is None:
            return self.row0(b) + j
        pt = self.page_table[b].cpu().to(torch.int64)
        return pt[j // self.page_size] * self.page_size + j % self.page_size


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, dtype, g, device, std=1.0):
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def make(cfg, device="cuda", *, n_kv_override=None, batch_override=None, n_tokens_override=None,
         parity_tails=False, quantized_keys=False, page_size=0) -> Workload:
    """Build configuration `cfg` (1-5 or "headline") on `device`.

    page_size: decode caches (indexer keys and latent) are stored in pages of
    this many rows, in a seeded random page order, addressed through a page
    table (name suffix "_paged"); 0 keeps them contiguous.
    quantized_keys: also store the decode indexer keys as a quantized cache
    (int8 codes + per-row f32 scales, idx_quantize_rows of the F16 keys); the
    workload's name gets the suffix "_q8" and the scorer reads the codes.

    Overrides shrink a configuration for parity tests that the oracle must
    finish quickly; they keep every other property (dtypes, heads, top_k,
    distributions, layout).
    """
    seed = 1000 + (cfg if isinstance(cfg, int) else 0)
    g = _gen(device, seed)
    dev = torch.device(device)
    i32 = dict(device=dev, dtype=torch.int32)

    if cfg == 1:
        n = n_tokens_override or 256
        T, B, H, d, top_k = n, 1, 4, 32, 64
        q = _randn((n, H, d), torch.float32, g, dev)
        k = _randn((n, d), torch.float32, g, dev)
        w = torch.rand((n, H), generator=g, device=dev, dtype=torch.float32)
        qa = _randn((n, 4, 32), torch.float32, g, dev)
        K = _randn((n, 1, 32), torch.float32, g, dev)
        V = _randn((n, 1, 32), torch.float32, g, dev)
        return Workload("tiny_prefill_fp32", "prefill", B, T, torch.tensor([n], **i32), [n], n, top_k, H, d,
                        q, w, k, 1 / math.sqrt(32), qa, K, V, 32, kv_seq_stride=n,
                        q_pos=torch.arange(n, **i32))

    if cfg in (2, 5, "headline"):
        H, d, top_k, Hq, dk, dv = 64, 128, 2048, 128, 576, 512
        if cfg == 2:
            B = batch_override or 8
            n_kv = [n_kv_override or 8192] * B
        elif cfg == "headline":
            B = batch_override or 64
            n_kv = [n_kv_override or 131072] * B
        else:
            B = batch_override or 64
            hi = n_kv_override or 131072
            lo = min(4096, hi)
            gh = torch.Generator().manual_seed(seed)
            n_kv = torch.randint(lo, hi + 1, (B,), generator=gh).tolist()
        max_n_kv = max(n_kv)
        if cfg == 5:
            starts = [0]
            for n in n_kv[:-1]:
                starts.append(starts[-1] + n)
            rows = starts[-1] + n_kv[-1]
            kv_start = torch.tensor(starts, **i32)
            stride = 0
        else:
            starts, kv_start, stride, rows = None, None, max_n_kv, B * max_n_kv
        q = _randn((B, H, d), torch.bfloat16, g, dev)
        w = _randn((B, H), torch.float32, g, dev, std=1 / math.sqrt(H))
        k = _randn((rows, d), torch.float16, g, dev)
        qa = _randn((B, Hq, dk), torch.bfloat16, g, dev)
        lat = _randn((rows, dk), torch.bfloat16, g, dev)
        name = {2: "decode_mla_8x8192", 5: "long_decode_mla_ragged", "headline": "decode_mla_64x131072"}[cfg]
        k8 = ks = None
        table = None
        if page_size:
            # logical page L = b * pages + lp goes to physical page perm[L]
            assert cfg != 5 and max_n_kv % page_size == 0, "paged workloads use equal, page-aligned sequences"
            pages = max_n_kv // page_size
            perm = torch.randperm(B * pages, generator=torch.Generator().manual_seed(seed)).to(dev)
            for name_t in ("k", "lat"):
                src = k if name_t == "k" else lat
                dst = torch.empty_like(src)
                dst.view(B * pages, page_size, -1)[perm] = src.view(B * pages, page_size, -1)
                if name_t == "k":
                    k = dst
                else:
                    lat = dst
            table = perm.view(B, pages).to(torch.int32)
            name += "_paged"
        if quantized_keys:
            # 128-byte code rows and a separate f32 scale array (the faster of the two layouts)
            from . import idx_quantize_rows
            k8, ks = idx_quantize_rows(k)
            name += "_q8"
        return Workload(name, "decode", B, 1, torch.tensor(n_kv, **i32), n_kv, max_n_kv, top_k, H, d, q, w, k,
                        1 / math.sqrt(192), qa, lat, None, dv, kv_start=kv_start, kv_start_host=starts,
                        kv_seq_stride=stride, k8=k8, k_scale=ks, page_table=table, page_size=page_size)

    if cfg == 3:
        n = n_tokens_override or 16384
        H, d, top_k, Hq, dk, dv = 64, 128, 2048, 128, 576, 512
        q = _randn((n, H, d), torch.bfloat16, g, dev)
        k = _randn((n, d), torch.bfloat16, g, dev)
        w = _randn((n, H), torch.float32, g, dev, std=1 / math.sqrt(H))
        qa = _randn((n, Hq, dk), torch.bfloat16, g, dev)
        lat = _randn((n, dk), torch.bfloat16, g, dev)
        return Workload(f"prefill_mla_{n}", "prefill", 1, n, torch.tensor([n], **i32), [n], n, top_k, H, d,
                        q, w, k, 1 / math.sqrt(192), qa, lat, None, dv, kv_seq_stride=n,
                        q_pos=torch.arange(n, **i32), hadamard=True)

    if cfg == 4:
        B = batch_override or 16
        base = n_kv_override or 32768
        n_kv = [base - 4 * s for s in range(B)] if parity_tails else [base] * B
        H, d, top_k, C = 32, 128, 2048, 64
        Hq, Hkv, dh = 32, 4, 128
        max_n_kv = max(n_kv)
        rows = B * max_n_kv
        q = _randn((B, H, d), torch.bfloat16, g, dev)
        w = _randn((B, H), torch.float32, g, dev, std=1 / math.sqrt(H))
        k = _randn((rows, d), torch.bfloat16, g, dev)
        qa = _randn((B, Hq, dh), torch.bfloat16, g, dev)
        K = _randn((rows, Hkv, dh), torch.bfloat16, g, dev)
        V = _randn((rows, Hkv, dh), torch.bfloat16, g, dev)
        return Workload("block_decode_gqa_16x32768", "block_decode", B, 1, torch.tensor(n_kv, **i32), n_kv,
                        max_n_kv, top_k, H, d, q, w, k, 1 / math.sqrt(dh), qa, K, V, dh,
                        kv_seq_stride=max_n_kv, block_size=C)

    raise ValueError(f"unknown config {cfg!r}")
