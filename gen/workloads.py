"""Seeded synthetic inputs for the decode sampling tail.

Shared by the tests, the bench and the smoke check.  This module holds none of
the tail's arithmetic: it only draws random inputs with the shapes and value
distributions of the workloads and rounds them to their storage formats.

Every array is a deterministic function of (workload name, seed, shape).  Large
weight matrices are drawn in independent 64-row chunks (one PCG64 stream per
chunk, keyed by ``SeedSequence([seed, stream, chunk])``) so they can be drawn
on several threads with identical bytes.
"""
from __future__ import annotations

import dataclasses
from concurrent.futures import ThreadPoolExecutor
import os

import numpy as np

# stream ids inside one seed
_S_HIDDEN, _S_GAMMA, _S_W, _S_PARAMS = 1, 2, 3, 4
_CHUNK_ROWS = 64


@dataclasses.dataclass
class Workload:
    name: str
    B: int
    H: int
    Hu: int
    V: int
    k: int
    eps: float
    zero_pad: int
    hidden_dtype: str          # "f32" | "f16" | "bf16"
    hidden: np.ndarray         # [B, H]: float32, or uint16 bit patterns for 16-bit dtypes
    gamma: np.ndarray          # [H] float32
    w_t: np.ndarray            # [H, V] uint16 bf16 bit patterns, V contiguous
    params: np.ndarray         # [B, 4] float32: top_k, top_p, temperature, u
    seed: int

    @property
    def hidden_bytes_per_elem(self) -> int:
        return 4 if self.hidden_dtype == "f32" else 2


def _rng(seed: int, stream: int, chunk: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, chunk])))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest even); returns uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).copy()
    t = (u >> np.uint32(16)) & np.uint32(1)
    t += np.uint32(0x7FFF)
    u += t
    u >>= np.uint32(16)
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16_matrix(seed: int, rows: int, cols: int, std: float, threads: int) -> np.ndarray:
    out = np.empty((rows, cols), dtype=np.uint16)
    nchunks = (rows + _CHUNK_ROWS - 1) // _CHUNK_ROWS

    def work(c: int) -> None:
        r0, r1 = c * _CHUNK_ROWS, min(rows, (c + 1) * _CHUNK_ROWS)
        a = _rng(seed, _S_W, c).standard_normal((r1 - r0) * cols, dtype=np.float32)
        a *= np.float32(std)
        out[r0:r1] = f32_to_bf16_bits(a).reshape(r1 - r0, cols)

    if threads <= 1 or nchunks == 1:
        for c in range(nchunks):
            work(c)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def _hidden(seed: int, B: int, H: int, dtype: str, row_scale=None):
    x = _rng(seed, _S_HIDDEN).standard_normal((B, H), dtype=np.float32)
    if row_scale is not None:
        x *= row_scale.astype(np.float32)[:, None]
    if dtype == "f32":
        return x
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    raise ValueError(dtype)


def _random_params(seed: int, B: int) -> np.ndarray:
    """top_k cycled {1, 50, 256} by row; top_p ~ U(0.5, 1); T ~ U(0.3, 1.5); u ~ U[0, 1)."""
    r = _rng(seed, _S_PARAMS)
    p = np.empty((B, 4), dtype=np.float32)
    p[:, 0] = np.array([1, 50, 256], dtype=np.float32)[np.arange(B) % 3]
    p[:, 1] = r.uniform(0.5, 1.0, B).astype(np.float32)
    p[:, 2] = r.uniform(0.3, 1.5, B).astype(np.float32)
    p[:, 3] = r.random(B, dtype=np.float32)
    return p


def pad_lanes(H: int, Hu: int) -> np.ndarray:
    """Interleaved pad layout used for padded hidden states: lane j is a pad when
    j % 16 == 15, filled from the front until H - Hu pads exist."""
    pads = np.zeros(H, dtype=bool)
    cand = np.nonzero(np.arange(H) % 16 == 15)[0][: H - Hu]
    pads[cand] = True
    assert pads.sum() == H - Hu, "layout needs H - Hu <= H / 16"
    return pads


def custom(B: int, H: int, V: int, k: int, *, hidden_dtype: str = "bf16", Hu: int | None = None,
           zero_pad: int = 1, eps: float = 1e-5, seed: int = 100, w_std: float = 0.02,
           dup_cols: int = 1, row_scale=None, params: np.ndarray | None = None,
           threads: int | None = None, name: str | None = None) -> Workload:
    """A synthetic tail input of any shape (same distributions as the named workloads).

    Hu < H with zero_pad=1 places zero pad lanes (x, gamma and W rows) at the
    interleaved positions of ``pad_lanes``; with zero_pad=0 the lanes [Hu, H) are
    simply not part of the hidden state and keep whatever was drawn.  dup_cols > 1 repeats each drawn W column that many times
    consecutively, planting exact logit ties.
    """
    threads = threads or min(16, os.cpu_count() or 1)
    Hu = H if Hu is None else Hu
    if V % dup_cols:
        raise ValueError("V must be a multiple of dup_cols")
    x = _hidden(seed, B, H, hidden_dtype, row_scale)
    gamma = _rng(seed, _S_GAMMA).uniform(0.5, 1.5, H).astype(np.float32)
    w = _normal_bf16_matrix(seed, H, V // dup_cols, w_std, threads)
    if dup_cols > 1:
        w = np.repeat(w, dup_cols, axis=1)
    if Hu < H and zero_pad:
        pads = pad_lanes(H, Hu)
        if hidden_dtype == "f32":
            x[:, pads] = 0.0
        else:
            x[:, pads] = 0  # +0.0 in both 16-bit formats
        gamma[pads] = 0.0
        w[pads, :] = 0
    p = _random_params(seed, B) if params is None else np.ascontiguousarray(params, np.float32)
    return Workload(name or f"custom_b{B}_h{H}_v{V}", B, H, Hu, V, k, eps, zero_pad, hidden_dtype,
                    np.ascontiguousarray(x), gamma, np.ascontiguousarray(w), p, seed)


# --------------------------------------------------------------------------- named workloads

def tiny(**kw) -> Workload:
    """gbs=1, H=256, V=4096, k=16; hidden fp32; params (16, 0.9, 0.7, 0.5); seed 0."""
    p = np.array([[16, 0.9, 0.7, 0.5]], dtype=np.float32)
    return custom(1, 256, 4096, 16, hidden_dtype="f32", seed=0, params=p, name="tiny", **kw)


def gptoss_g8(**kw) -> Workload:
    """GPT-OSS-shaped decode tail: gbs=8, H=2880, V=201088, k=256, hidden bf16; seed 1."""
    return custom(8, 2880, 201088, 256, hidden_dtype="bf16", seed=1, name="gptoss_g8", **kw)


def padded_g64(**kw) -> Workload:
    """gbs=64, H=3072, hidden_actual=2880, zero interleaved pads in x/gamma/W, hidden fp16;
    rows b % 4 == 0 greedy (temperature 0); seed 2."""
    B = 64
    p = _random_params(2, B)
    p[np.arange(B) % 4 == 0, 2] = 0.0
    return custom(B, 3072, 201088, 256, hidden_dtype="f16", Hu=2880, zero_pad=1, seed=2,
                  params=p, name="padded_g64", **kw)


def adversarial_g32(**kw) -> Workload:
    """gbs=32, H=2880, V=201088, k=256: W columns repeated in groups of 4 (exact ties),
    rows b % 8 == 1 scaled x1e3 and b % 8 == 2 scaled x1e-3 before rounding to bf16,
    params: rows r % 3 == 0 top_k=1, r % 3 == 1 top_p=1.0, r % 3 == 2 temperature=5.0,
    u = 0.0 on even rows and 0.999999 on odd rows; seed 3."""
    B = 32
    scale = np.ones(B, dtype=np.float32)
    scale[np.arange(B) % 8 == 1] = 1e3
    scale[np.arange(B) % 8 == 2] = 1e-3
    p = _random_params(3, B)
    r = np.arange(B)
    p[r % 3 == 0, 0] = 1.0
    p[r % 3 == 1, 1] = 1.0
    p[r % 3 == 2, 2] = 5.0
    p[:, 3] = np.where(r % 2 == 0, np.float32(0.0), np.float32(0.999999))
    return custom(B, 2880, 201088, 256, hidden_dtype="bf16", seed=3, dup_cols=4,
                  row_scale=scale, params=p, name="adversarial_g32", **kw)


def large_g1024(**kw) -> Workload:
    """gbs=1024, H=2880, V=201088, k=256, hidden bf16, random params; seed 4."""
    return custom(1024, 2880, 201088, 256, hidden_dtype="bf16", seed=4, name="large_g1024", **kw)


NAMED = {
    "tiny": tiny,
    "gptoss_g8": gptoss_g8,
    "padded_g64": padded_g64,
    "adversarial_g32": adversarial_g32,
    "large_g1024": large_g1024,
}


def make(name: str, **kw) -> Workload:
    return NAMED[name](**kw)
