"""Seeded synthetic inputs for the tensor-parallel sharded linear pipeline.

This module is shared by the oracle-side tests and by the CUDA-side tests and
bench. It holds no arithmetic of the method (no products, sums, activations or
shard layouts): it only draws numbers and rounds them to the storage type the
GPU reads, so that both sides start from identical values.

Value distributions follow the workloads the pages describe: integer-valued
inputs for the exact case, N(0, 1) activations and small-variance normal
weights for the LLaMA-shaped cases. Weights use the [in, out] orientation the
pages use (Y = X @ W).

Generation is chunked: a shape is filled from ``CHUNKS`` independent PCG64
streams spawned from one ``SeedSequence(seed)``, so the values depend only on
(seed, shape, distribution) and not on the thread count.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

CHUNKS = 64
_THREADS = max(1, min(16, os.cpu_count() or 1))


def _fill(seed: int, n: int, kind: str, a: float, b: float) -> np.ndarray:
    out = np.empty(n, np.float32)
    seqs = np.random.SeedSequence(seed).spawn(CHUNKS)

    def work(i: int) -> None:
        lo, hi = i * n // CHUNKS, (i + 1) * n // CHUNKS
        if hi <= lo:
            return
        r = np.random.Generator(np.random.PCG64(seqs[i]))
        o = out[lo:hi]
        if kind == "normal":
            r.standard_normal(hi - lo, dtype=np.float32, out=o)
            if a != 1.0:
                o *= np.float32(a)
            to_bf16_inplace(o)
        elif kind == "int":
            o[:] = r.integers(int(a), int(b) + 1, size=hi - lo, dtype=np.int32)
        elif kind == "uniform":
            r.random(hi - lo, dtype=np.float32, out=o)
            o *= np.float32(b - a)
            o += np.float32(a)
        else:  # pragma: no cover - internal misuse
            raise ValueError(kind)

    if n >= (1 << 20):
        with ThreadPoolExecutor(_THREADS) as ex:
            list(ex.map(work, range(CHUNKS)))
    else:
        for i in range(CHUNKS):
            work(i)
    return out


def to_bf16_inplace(a: np.ndarray) -> np.ndarray:
    """Round a float32 array to the nearest bfloat16 value (ties to even), in place.

    The result is still float32 storage, but every value is exactly
    representable in bfloat16, so a later cast to bf16 is exact. Inputs are
    finite normals here; NaN/Inf handling is not needed.
    """
    u = a.view(np.uint32)
    t = u >> np.uint32(16)
    t &= np.uint32(1)
    t += np.uint32(0x7FFF)
    u += t
    u &= np.uint32(0xFFFF0000)
    return a


def normal(seed: int, shape, std: float = 1.0) -> np.ndarray:
    """N(0, std^2) values rounded to bfloat16, returned as float32."""
    n = int(np.prod(shape))
    return _fill(seed, n, "normal", std, 0.0).reshape(shape)


def uniform_ints(seed: int, shape, lo: int = -3, hi: int = 3) -> np.ndarray:
    """Integers uniform on {lo, ..., hi}, stored as float32."""
    n = int(np.prod(shape))
    return _fill(seed, n, "int", lo, hi).reshape(shape)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """The upper 16 bits of bf16-representable float32 values (the bf16 encoding)."""
    return (a.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# ---------------------------------------------------------------------------
# Workloads
# ---------------------------------------------------------------------------

def worked_example():
    """X = [10, 20] and the 2x4 weight W = [[1,2,3,4],[5,6,7,8]] of the
    worked example on the "CUDA tensor parallel computations" page (section
    on the minimal matrix-multiply foundation)."""
    X = np.array([[10, 20]], np.float32)
    W = np.array([[1, 2, 3, 4], [5, 6, 7, 8]], np.float32)
    return X, W


def int_mlp(T: int = 16, H: int = 64, I: int = 256, seed: int = 0):
    """Exact-integer MLP: X[T,H], W1[H,I], W2[I,H] uniform on {-3..3}."""
    return dict(
        X=uniform_ints(seed * 1000 + 1, (T, H)),
        W1=uniform_ints(seed * 1000 + 2, (H, I)),
        W2=uniform_ints(seed * 1000 + 3, (I, H)),
    )


def swiglu_mlp(T: int, H: int, I: int, seeds=(1, 2, 3, 4), std: float = 0.02):
    """LLaMA-shaped SwiGLU MLP: X~N(0,1), Wg, Wu [H,I], Wd [I,H] ~ N(0, std^2)."""
    sx, sg, su, sd = seeds
    return dict(
        X=normal(sx, (T, H)),
        Wg=normal(sg, (H, I), std),
        Wu=normal(su, (H, I), std),
        Wd=normal(sd, (I, H), std),
    )


def mlp_backward(T: int, H: int, I: int, seeds=(1, 2, 3, 4, 40), std: float = 0.02):
    """The SwiGLU MLP's inputs plus an output gradient dY ~ N(0,1) [T,H]."""
    d = swiglu_mlp(T, H, I, seeds[:4], std)
    d["dY"] = normal(seeds[4], (T, H))
    return d


def token_ids(seed: int, T: int, V: int) -> np.ndarray:
    """Token ids (or labels) uniform on {0, ..., V-1}, int32."""
    return uniform_ints(seed, (T,), 0, V - 1).astype(np.int32)


def vocab_lm(T: int, H: int, V: int, seeds=(50, 51, 52, 53), std: float = 0.02):
    """A zero-block language model's ends: embedding table E [V,H] ~ N(0,1),
    LM head W [H,V] ~ N(0, std^2), input ids and next-token labels [T]."""
    se, sw, si, sl = seeds
    return dict(E=normal(se, (V, H)), W_lm=normal(sw, (H, V), std), ids=token_ids(si, T, V),
                labels=token_ids(sl, T, V))


def moe_routing(seed: int, T: int, E: int, k: int):
    """Synthetic top-k routing: for each token k distinct experts (the first
    uniform on {0..E-1}, each next one a uniform nonzero step further,
    modulo E, moved on past experts the token already has) and k weights
    uniform on [0.05, 1), fp32."""
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    first = uniform_ints(seed, (T,), 0, E - 1).astype(np.int64)
    ids = np.empty((T, k), dtype=np.int64)
    ids[:, 0] = first
    taken = [first]
    for j in range(1, k):
        step = uniform_ints(seed + 1000 * j, (T,), 1, max(E - 1, 1)).astype(np.int64)
        cand = (ids[:, j - 1] + step) % E
        for _ in range(E):
            clash = np.zeros(T, dtype=bool)
            for prev in taken:
                clash |= cand == prev
            if not clash.any():
                break
            cand = np.where(clash, (cand + 1) % E, cand)
        ids[:, j] = cand
        taken.append(cand)
    w = _fill(seed + 7, T * k, "uniform", 0.05, 1.0).reshape(T, k).astype(np.float32)
    return ids.astype(np.int32), w


def moe_experts(E: int, H: int, I: int, seed: int = 60, std: float = 0.02):
    """E SwiGLU experts: Wg, Wu [H,I], Wd [I,H] ~ N(0, std^2)."""
    return [dict(W1=normal(seed + 3 * e, (H, I), std), W_up=normal(seed + 3 * e + 1, (H, I), std),
                 W2=normal(seed + 3 * e + 2, (I, H), std)) for e in range(E)]


def gqa_proj(T: int, H: int, hq: int, hkv: int, hd: int, seeds=(5, 6, 7, 8, 9),
             std: float = 0.02):
    """Attention projections: X~N(0,1); Wq [H, hq*hd], Wk, Wv [H, hkv*hd],
    Wo [hq*hd, H] ~ N(0, std^2)."""
    sx, sq, sk, sv, so = seeds
    return dict(
        X=normal(sx, (T, H)),
        Wq=normal(sq, (H, hq * hd), std),
        Wk=normal(sk, (H, hkv * hd), std),
        Wv=normal(sv, (H, hkv * hd), std),
        Wo=normal(so, (hq * hd, H), std),
    )


def decode_mlp(T: int, H: int = 8192, I: int = 28672, seed: int = 10,
               std: float = 0.015):
    """Decode-shaped SwiGLU MLP: few tokens, 70B-like H and I."""
    return dict(
        X=normal(seed * 1000 + 1, (T, H)),
        Wg=normal(seed * 1000 + 2, (H, I), std),
        Wu=normal(seed * 1000 + 3, (H, I), std),
        Wd=normal(seed * 1000 + 4, (I, H), std),
    )


def stack(T: int, H: int = 4096, I: int = 11008, hq: int = 32, hkv: int = 8,
          hd: int = 128, V: int = 32000, layers: int = 4, std: float = 0.02):
    """Inputs of the 4-block stack: X, per-layer attention and MLP weights
    (seeds 11.. onward, 7 matrices per layer) and the LM head (seed 39 for
    4 layers). Norm gains are 1."""
    out = dict(X=normal(11 * 1000, (T, H)), layers=[])
    s = 11
    for _ in range(layers):
        L = dict(
            Wq=normal(s, (H, hq * hd), std), Wk=normal(s + 1, (H, hkv * hd), std),
            Wv=normal(s + 2, (H, hkv * hd), std), Wo=normal(s + 3, (hq * hd, H), std),
            Wg=normal(s + 4, (H, I), std), Wu=normal(s + 5, (H, I), std),
            Wd=normal(s + 6, (I, H), std),
        )
        out["layers"].append(L)
        s += 7
    out["W_lm"] = normal(s, (H, V), std)
    return out
