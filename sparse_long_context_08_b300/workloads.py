"""Seeded synthetic decode workloads for the EntmaxKV paged-KV pipeline.

This module only produces inputs: queries, a paged K/V pool, a page table and
sequence lengths, with the sizes and value distributions of the five decode
workloads (tiny, GQA 32K, batched 128K, 1M, Gaussian-selection 64K). It holds
none of the method's arithmetic (no scores, bounds, thresholds or attention);
the same arrays feed both the CPU oracle and the CUDA library.

Recipe (all draws from numpy PCG64 streams spawned from one SeedSequence):

* q ~ N(0, 1), fp32, shape [B, Hq, d].
* Keys of a (physical block, kv head) page: k_t = c_page + eps_scale * e_t with
  e_t ~ N(0, I).  Background cluster means c_page ~ N(0, cluster_std^2 I).
* Planted pages (per sequence and kv head, logical pages chosen uniformly
  without replacement): c_page = planted_scale * u, u = unit vector of the mean
  of that kv head's query group.  These are the "high-score pages".
* "Flat" kv heads (Gaussian workload): c_page = 0 and eps_scale = flat_eps.
* V ~ N(0, 1).
* page_table: a random permutation of all physical blocks laid out [B, NP];
  entries past a sequence's last page are -1.
* K/V in bf16 are stored as uint16 bit patterns, rounded to nearest-even from
  the fp32 draw.

Sizes follow the paged layout [num_blocks, Hkv, P, d] with one (block, head)
page contiguous.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
import os

import numpy as np

# ---------------------------------------------------------------------------
# Named workloads.  Sizes are the decode configurations the library is
# measured on; every field can be overridden (smaller sizes for parity tests).
# ---------------------------------------------------------------------------
CONFIGS: dict[str, dict] = {
    # batch 1, 1 head, d=64, 4096 tokens, page 16, fp32, scale 4/sqrt(d),
    # alpha 1.5, 32 pages (512 tokens) kept.
    "tiny": dict(batch=1, num_q_heads=1, num_kv_heads=1, head_dim=64,
                 context=4096, page_size=16, dtype="f32",
                 scale_mult=4.0, alpha=1.5, policy="topk",
                 budget_tokens=512, seed=0),
    # Llama-style GQA decode: 32 q / 8 kv heads, d=128, 32K tokens, page 16,
    # bf16, alpha 1.5, 2048-token budget (128 pages).
    "gqa32k": dict(batch=1, num_q_heads=32, num_kv_heads=8, head_dim=128,
                   context=32768, page_size=16, dtype="bf16",
                   alpha=1.5, policy="topk", budget_tokens=2048, seed=1),
    # Batched long context: batch 8, 128K tokens, page 32, 8 planted
    # high-score pages per (sequence, kv head), budget 4096 tokens.
    "long128k": dict(batch=8, num_q_heads=32, num_kv_heads=8, head_dim=128,
                     context=131072, page_size=32, dtype="bf16",
                     alpha=1.5, policy="topk", budget_tokens=4096,
                     planted_pages=8, planted_scale=8.0, seed=2),
    # Very long context: batch 1, 1M tokens, page 32; clustered keys with 48
    # planted pages per kv head so that the entmax support stays within a few
    # dozen pages.
    "ctx1m": dict(batch=1, num_q_heads=32, num_kv_heads=8, head_dim=128,
                  context=1048576, page_size=32, dtype="bf16",
                  alpha=1.5, policy="topk", budget_tokens=4096,
                  eps_scale=0.5, planted_pages=48, planted_scale=10.0,
                  seed=3),
    # Gaussian-aware selection: batch 16, 64K tokens, page 16; kv heads 0-3
    # sharp (planted pages), 4-7 flat (k = 0.25 e); tau-hat policy with margin
    # 0.1 and a cap of 8192 tokens (512 pages).
    "gauss64k": dict(batch=16, num_q_heads=32, num_kv_heads=8, head_dim=128,
                     context=65536, page_size=16, dtype="bf16",
                     alpha=1.5, policy="gauss", budget_tokens=8192,
                     delta=0.1, planted_pages=8, planted_scale=8.0,
                     flat_heads=(4, 5, 6, 7), flat_eps=0.25, seed=4),
}

_DEFAULTS = dict(scale_mult=1.0, cluster_std=0.5, eps_scale=1.0,
                 planted_pages=0, planted_scale=8.0, flat_heads=(),
                 flat_eps=0.25, delta=0.0, seq_lens=None)

_CHUNK_ELEMS = 1 << 20  # elements per independent RNG stream for K/V draws


@dataclass
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    dtype: str                 # "f32" or "bf16"
    scale: np.float32          # score scale s (z = s * q.k)
    alpha: float
    policy: str                # "topk", "gauss" or "topk_shared"
    budget_tokens: int
    delta: float
    seq_lens: np.ndarray       # int32 [B]
    max_pages: int
    num_blocks: int
    q: np.ndarray              # fp32 [B, Hq, d]
    k_pool: np.ndarray         # fp32 or uint16(bf16 bits) [nb, Hkv, P, d]
    v_pool: np.ndarray
    page_table: np.ndarray     # int32 [B, max_pages], -1 past the end
    planted: np.ndarray        # int32 [B, Hkv, n_planted] logical page ids
    seed: int
    params: dict = field(default_factory=dict)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def cap_pages(self) -> int:
        return self.budget_tokens // self.page_size

    def pages_of(self, b: int) -> int:
        return -(-int(self.seq_lens[b]) // self.page_size)


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even) and return the uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).copy()
    u += np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (u >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _fill_pool(out: np.ndarray, seq: np.random.SeedSequence, bf16: bool,
               mean: np.ndarray | None, eps_scale: np.ndarray) -> None:
    """out[blk, h, t, :] = mean[blk, h, :] + eps_scale[h] * N(0, 1) draws.

    Draws are made in fixed chunks of whole blocks, each chunk with its own
    spawned stream, so the result does not depend on the thread count.
    """
    nb, hkv, P, d = out.shape
    per_block = hkv * P * d
    blocks_per_chunk = max(1, _CHUNK_ELEMS // per_block)
    n_chunks = -(-nb // blocks_per_chunk)
    children = seq.spawn(n_chunks)
    scale = np.asarray(eps_scale, dtype=np.float32).reshape(1, hkv, 1, 1)

    def work(i: int) -> None:
        b0 = i * blocks_per_chunk
        b1 = min(nb, b0 + blocks_per_chunk)
        g = np.random.Generator(np.random.PCG64(children[i]))
        x = g.standard_normal((b1 - b0, hkv, P, d), dtype=np.float32)
        x *= scale
        if mean is not None:
            x += mean[b0:b1, :, None, :]
        out[b0:b1] = bf16_bits_from_f32(x) if bf16 else x

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, range(n_chunks)))


def make_workload(name: str, **overrides) -> Workload:
    """Build the named workload; keyword overrides replace any config field.

    Useful overrides: batch, context, seq_lens (list of per-sequence lengths,
    ragged allowed), num_q_heads, num_kv_heads, head_dim, page_size, dtype,
    alpha, budget_tokens, delta, planted_pages, seed.
    """
    if name not in CONFIGS:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(CONFIGS)}")
    cfg = dict(_DEFAULTS)
    cfg.update(CONFIGS[name])
    cfg.update(overrides)

    B = int(cfg["batch"])
    Hq = int(cfg["num_q_heads"])
    Hkv = int(cfg["num_kv_heads"])
    d = int(cfg["head_dim"])
    P = int(cfg["page_size"])
    if Hq % Hkv:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    G = Hq // Hkv
    if cfg["seq_lens"] is None:
        seq_lens = np.full(B, int(cfg["context"]), dtype=np.int32)
    else:
        seq_lens = np.asarray(cfg["seq_lens"], dtype=np.int32)
        if seq_lens.shape != (B,):
            raise ValueError("seq_lens must have one entry per sequence")
    pages = [-(-int(n) // P) for n in seq_lens]
    max_pages = max(1, max(pages))
    num_blocks = int(sum(pages))
    bf16 = cfg["dtype"] == "bf16"
    scale = np.float32(cfg["scale_mult"] / math.sqrt(d))

    root = np.random.SeedSequence(int(cfg["seed"]))
    s_q, s_c, s_perm, s_plant, s_k, s_v = root.spawn(6)

    q = np.random.Generator(np.random.PCG64(s_q)).standard_normal(
        (B, Hq, d), dtype=np.float32)

    # Physical block ids: a random permutation laid out per sequence.
    perm = np.random.Generator(np.random.PCG64(s_perm)).permutation(num_blocks).astype(np.int32)
    page_table = np.full((B, max_pages), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        page_table[b, :pages[b]] = perm[off:off + pages[b]]
        off += pages[b]

    # Per-(block, kv head) cluster means.
    flat = set(int(h) for h in cfg["flat_heads"])
    mean = (np.random.Generator(np.random.PCG64(s_c)).standard_normal(
        (num_blocks, Hkv, d), dtype=np.float32) * np.float32(cfg["cluster_std"]))
    for h in flat:
        mean[:, h, :] = 0.0
    eps_scale = np.array([cfg["flat_eps"] if h in flat else cfg["eps_scale"]
                          for h in range(Hkv)], dtype=np.float32)

    n_pl = int(cfg["planted_pages"])
    planted = np.zeros((B, Hkv, n_pl), dtype=np.int32)
    if n_pl:
        gp = np.random.Generator(np.random.PCG64(s_plant))
        for b in range(B):
            for h in range(Hkv):
                if h in flat:
                    planted[b, h, :] = -1
                    continue
                pick = np.sort(gp.choice(pages[b], size=min(n_pl, pages[b]), replace=False))
                planted[b, h, :len(pick)] = pick
                u = q[b, h * G:(h + 1) * G].astype(np.float64).mean(axis=0)
                u /= np.linalg.norm(u)
                blk = page_table[b, pick]
                mean[blk, h, :] = (float(cfg["planted_scale"]) * u).astype(np.float32)

    pool_dtype = np.uint16 if bf16 else np.float32
    k_pool = np.empty((num_blocks, Hkv, P, d), dtype=pool_dtype)
    v_pool = np.empty((num_blocks, Hkv, P, d), dtype=pool_dtype)
    _fill_pool(k_pool, s_k, bf16, mean, eps_scale)
    del mean
    _fill_pool(v_pool, s_v, bf16, None, np.ones(Hkv, dtype=np.float32))

    return Workload(
        name=name, batch=B, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
        page_size=P, dtype=cfg["dtype"], scale=scale, alpha=float(cfg["alpha"]),
        policy=cfg["policy"], budget_tokens=int(cfg["budget_tokens"]),
        delta=float(cfg["delta"]), seq_lens=seq_lens, max_pages=max_pages,
        num_blocks=num_blocks, q=q, k_pool=k_pool, v_pool=v_pool,
        page_table=page_table, planted=planted, seed=int(cfg["seed"]),
        params={k: cfg[k] for k in ("cluster_std", "eps_scale", "planted_pages",
                                    "planted_scale", "flat_eps", "scale_mult")}
        | {"flat_heads": sorted(flat), "context": int(max(seq_lens))},
    )
