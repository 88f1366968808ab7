"""Seeded synthetic inputs for the chunk-forward kkt_solve step of Gated DeltaNet.

This module is shared by the tests, the benchmark and the oracle's callers.  It
only draws inputs; it contains none of the method's arithmetic (no Gram matrix,
no gate factor, no inverse).

Recipe (the published workloads are not available, these stand in for them;
the shapes are the ones quoted on the MindSpeed-Ops PR page "feat(triton): add
chunk_gated_delta_rule_fwd_kkt_solve", performance table):
  * k    ~ N(0, 1) in fp32, L2-normalised over the head dimension K for every
           (token, head), then rounded to bf16 (round-to-nearest-even), or to
           fp16 for the fp16-input variants, or kept in fp32 for the fp32-key
           variants.
  * beta = sigmoid(N(0, 1)), rounded to bf16 (or fp16, or kept fp32).
  * g    = per-token U(-0.1, 0) log-decay in fp32, summed inclusively inside
           every chunk (64 tokens, or 128 for the chunk-128 variants); the sum
           restarts at each chunk start, and chunks restart at every sequence
           start.
  * varlen: 8 packed sequences with integer lengths ~ U[100, 4000], redrawn
           from the same generator until the total is at most 16384;
           cu_seqlens = [0, cumsum(lengths)] as int32 and k is [1, T, H, K].
All draws use numpy's PCG64 generator seeded with the workload's seed, so the
bytes are identical on every platform.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

CHUNK = 64


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int            # batch size, or the number of sequences when varlen
    T: int            # tokens per sequence, or total packed tokens when varlen
    H: int
    K: int
    out_dtype: str    # "f32", "bf16" or "f16"
    seed: int
    varlen_lengths: Optional[tuple] = None   # per-sequence lengths when packed
    use_g: bool = True
    use_beta: bool = True
    k_dtype: str = "bf16"       # "bf16" or "f16": type k is rounded to; "f32": kept
    beta_dtype: str = "bf16"    # "bf16", "f16" or "f32"
    chunk: int = CHUNK          # chunk length the log-gate's running sum restarts at

    @property
    def token_heads(self) -> int:
        return self.B * self.T * self.H if self.varlen_lengths is None else self.T * self.H

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _varlen_lengths(seed: int, n: int = 8, lo: int = 100, hi: int = 4000, cap: int = 16384):
    rng = np.random.default_rng(seed)
    while True:
        lens = rng.integers(lo, hi + 1, size=n)
        if int(lens.sum()) <= cap:
            return tuple(int(x) for x in lens)


def varlen_workload(name: str, seed: int, H: int = 16, K: int = 128, out_dtype: str = "f32",
                    n: int = 8, lo: int = 100, hi: int = 4000, cap: int = 16384) -> Workload:
    lens = _varlen_lengths(seed, n, lo, hi, cap)
    return Workload(name, B=len(lens), T=int(sum(lens)), H=H, K=K, out_dtype=out_dtype,
                    seed=seed, varlen_lengths=lens)


# The workloads, named by their shapes; seeds 1 to 5.
CONFIGS = {
    "B1_T256_H8_K128": Workload("B1_T256_H8_K128", 1, 256, 8, 128, "f32", seed=1),
    "B2_T2000_H5_K128": Workload("B2_T2000_H5_K128", 2, 2000, 5, 128, "f32", seed=2),
    "B1_T8192_H8_K128": Workload("B1_T8192_H8_K128", 1, 8192, 8, 128, "bf16", seed=3),
    "varlen8_H16_K128": varlen_workload("varlen8_H16_K128", seed=4),
    "B2_T16384_H32_K128": Workload("B2_T16384_H32_K128", 2, 16384, 32, 128, "bf16", seed=5),
}


def cu_seqlens_of(wl: Workload) -> Optional[np.ndarray]:
    if wl.varlen_lengths is None:
        return None
    return np.concatenate([[0], np.cumsum(wl.varlen_lengths)]).astype(np.int32)


def _sequence_bounds(wl: Workload):
    """(start, end) token rows of every sequence in the flattened token axis."""
    if wl.varlen_lengths is None:
        return [(b * wl.T, (b + 1) * wl.T) for b in range(wl.B)]
    cu = cu_seqlens_of(wl)
    return [(int(cu[n]), int(cu[n + 1])) for n in range(wl.B)]


def _chunk_local_cumsum(a: np.ndarray, bounds, chunk: int = CHUNK) -> np.ndarray:
    """Inclusive running sum of a [Ntok, H] restarted at every chunk start."""
    g = np.empty_like(a)
    for s, e in bounds:
        for c0 in range(s, e, chunk):
            c1 = min(c0 + chunk, e)
            g[c0:c1] = np.cumsum(a[c0:c1], axis=0, dtype=np.float32)
    return g


def make_inputs(wl: Workload):
    """Returns a dict of CPU tensors: k (bf16 or fp16), g (fp32 or None), beta
    (bf16, fp16, fp32 or None), cu_seqlens (int32 or None).  Fixed-length k is [B, T, H, K]; packed
    (varlen) k is [1, T, H, K]."""
    rng = np.random.default_rng(wl.seed)
    ntok = wl.B * wl.T if wl.varlen_lengths is None else wl.T
    H, K = wl.H, wl.K
    k = np.empty((ntok, H, K), dtype=np.float32)
    step = max(1, (1 << 24) // (H * K))          # draw in slices to bound memory
    for r0 in range(0, ntok, step):
        r1 = min(ntok, r0 + step)
        x = rng.standard_normal((r1 - r0, H, K), dtype=np.float32)
        x /= np.sqrt(np.sum(x * x, axis=-1, keepdims=True, dtype=np.float32))
        k[r0:r1] = x
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((ntok, H), dtype=np.float32)))
    a = -0.1 * rng.random((ntok, H), dtype=np.float32)
    g = _chunk_local_cumsum(a.astype(np.float32), _sequence_bounds(wl), wl.chunk)

    lead = (wl.B, wl.T) if wl.varlen_lengths is None else (1, wl.T)
    types = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}
    kt = torch.from_numpy(k).to(types[wl.k_dtype]).reshape(*lead, H, K)
    out = {
        "k": kt,
        "g": torch.from_numpy(g).reshape(*lead, H) if wl.use_g else None,
        "beta": torch.from_numpy(beta.astype(np.float32)).to(types[wl.beta_dtype]).reshape(*lead, H)
        if wl.use_beta else None,
        "cu_seqlens": None,
    }
    cu = cu_seqlens_of(wl)
    if cu is not None:
        out["cu_seqlens"] = torch.from_numpy(cu)
    return out


def tile_list(wl: Workload):
    """All (sequence, chunk, head) tiles of a workload with their token ranges:
    list of (n, c, h, row0, L) where row0 is the first token row of the chunk in
    the flattened token axis and L <= wl.chunk its length."""
    tiles = []
    for n, (s, e) in enumerate(_sequence_bounds(wl)):
        for c, r0 in enumerate(range(s, e, wl.chunk)):
            L = min(wl.chunk, e - r0)
            for h in range(wl.H):
                tiles.append((n, c, h, r0, L))
    return tiles


def sample_tiles(wl: Workload, count: int, seed: int = 1234):
    """A seeded sample of tiles that always includes the first and last tile and
    every partial (shorter than 64) chunk of head 0 and the last head."""
    tiles = tile_list(wl)
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(len(tiles), size=min(count, len(tiles)), replace=False).tolist())
    pick.update({0, len(tiles) - 1})
    for i, t in enumerate(tiles):
        if t[4] < CHUNK and t[2] in (0, wl.H - 1):
            pick.add(i)
    return [tiles[i] for i in sorted(pick)]
