"""Seeded synthetic inputs for the attention path.

This module holds no arithmetic of the method: it only draws random numbers
and rounds them to binary16.  Both the CUDA path's tests and benchmark and
the CPU oracle read the arrays it returns.

Recipe: config ``k`` uses seed ``k``.  One numpy ``PCG64(seed)`` stream draws,
in order: the per-sequence lengths (variable-length workload only, uniform
integers in [256, 4096]), then Q, K, V^T and dO as standard-normal binary32
in the boundary layouts, with Q multiplied by its standard deviation where
the workload asks for a sharper softmax.  Everything is rounded to binary16
(round to nearest even, numpy's ``astype``).

Layouts: q, dout [B][H][T][64]; k [B][Hkv][T][64]; vt [B][Hkv][64][T].
"""
from dataclasses import dataclass
from typing import Optional

import numpy as np

HEAD_DIM = 64
SCALE = 0.125


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seq: int
    heads: int
    kv_heads: int
    causal: bool
    varlen: bool = False
    q_std: float = 1.0
    len_lo: int = 256
    len_hi: int = 4096
    seed: int = 0
    scale: float = SCALE

    @property
    def group(self) -> int:
        return self.heads // self.kv_heads


# The five workloads of the method's evaluation: shapes and value
# distributions as the target configurations state them.
WORKLOADS = {
    1: Workload("causal T=128 H=2 Hkv=1 d=64", 1, 128, 2, 1, True, seed=1),
    2: Workload("causal T=1024 H=8 Hkv=8 d=64", 1, 1024, 8, 8, True, seed=2),
    3: Workload("causal GQA T=4096 H=32 Hkv=8 d=64 Q~N(0,16)", 1, 4096, 32, 8, True,
                q_std=4.0, seed=3),
    4: Workload("non-causal varlen B=16 len~U[256,4096] pad 4096 H=16 Hkv=16 d=64",
                16, 4096, 16, 16, False, varlen=True, seed=4),
    5: Workload("causal GQA T=16384 H=32 Hkv=4 d=64", 1, 16384, 32, 4, True, seed=5),
}


def make_inputs(w: Workload, seed: Optional[int] = None) -> dict:
    """Draw q, k, vt, dout (binary16) and lens (int32 or None) for ``w``."""
    rng = np.random.Generator(np.random.PCG64(w.seed if seed is None else seed))
    lens = None
    if w.varlen:
        lens = rng.integers(w.len_lo, w.len_hi, size=w.batch, endpoint=True).astype(np.int32)
    B, H, Hkv, T, d = w.batch, w.heads, w.kv_heads, w.seq, HEAD_DIM
    q = rng.standard_normal((B, H, T, d), dtype=np.float32)
    k = rng.standard_normal((B, Hkv, T, d), dtype=np.float32)
    vt = rng.standard_normal((B, Hkv, d, T), dtype=np.float32)
    dout = rng.standard_normal((B, H, T, d), dtype=np.float32)
    if w.q_std != 1.0:
        q *= np.float32(w.q_std)
    return dict(q=q.astype(np.float16), k=k.astype(np.float16),
                vt=vt.astype(np.float16), dout=dout.astype(np.float16), lens=lens)


def custom(batch, seq, heads, kv_heads, causal=True, lens=None, q_std=1.0, seed=0,
           name="custom") -> Workload:
    """A small workload for edge-case tests; ``lens`` fixes the lengths if given."""
    return Workload(name, batch, seq, heads, kv_heads, causal, varlen=False,
                    q_std=q_std, seed=seed)


def make_custom_inputs(batch, seq, heads, kv_heads, *, causal=True, lens=None,
                       q_std=1.0, seed=0) -> dict:
    """Inputs for an arbitrary small shape, lengths given explicitly (or None)."""
    w = custom(batch, seq, heads, kv_heads, causal, q_std=q_std, seed=seed)
    out = make_inputs(w)
    out["lens"] = None if lens is None else np.asarray(lens, dtype=np.int32)
    return out
