"""Seeded synthetic inputs for the DeepSeek V4.1 Engram forward path.

This module is shared by the CUDA path's tests and benchmark and by the oracle's tests. It holds
none of the method's arithmetic: it draws token ids, hash tables, fp8 table rows, activations and
weights with numpy's PCG64 generator and casts them to their storage types (bf16, float8_e4m3fn)
through torch's own dtype casts. Nothing here hashes, gathers, projects or gates.

Every array is returned as raw storage bits in numpy: bf16 as ``uint16``, fp8 e4m3 and e8m0 as
``uint8``, ids as ``int32``, hash-table constants as ``uint64``/``int64``.

Value distributions follow the fixture rules named in the engram module docs ("Module engram",
CPU reference; functions ``regen_bf16_matrix``: scale in^-0.5; ``regen_bf16_qk``: 1 +- 0.05;
``regen_table``: fp8 table with e8m0 block scales) and the workload list of the Engram pages
(dim 5120, hc 4, 24 rows per position, head_dim 64).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

BASE_SEED = 0x5EED
SCALE_BLOCK = 32  # e8m0 block size along head_dim


@dataclasses.dataclass(frozen=True)
class Geometry:
    """Shapes of one Engram layer and of its hash tables."""

    dim: int
    hc_mult: int
    n_heads: int
    max_ngram_size: int
    head_dim: int
    vocab: int          # tokenizer vocabulary (token ids are drawn from it)
    n_compressed: int   # size of the compressed vocabulary the token map targets
    prime_floor: int    # per-slot primes are the consecutive primes >= this

    @property
    def n_hash_cols(self) -> int:
        return (self.max_ngram_size - 1) * self.n_heads

    @property
    def K(self) -> int:  # wkv input width
        return self.n_hash_cols * self.head_dim

    @property
    def N(self) -> int:  # wkv output width
        return self.dim * (self.hc_mult + 1)


# Tiny geometry: dim 256, head_dim 32, vocab 1000 -> 512 compressed ids, primes from 1009.
TINY = Geometry(dim=256, hc_mult=4, n_heads=8, max_ngram_size=4, head_dim=32,
                vocab=1000, n_compressed=512, prime_floor=1009)
# Full width: dim 5120, hc 4, head_dim 64, vocab 129280, primes from 2^19 (~805 MB fp8 table).
FULL = Geometry(dim=5120, hc_mult=4, n_heads=8, max_ngram_size=4, head_dim=64,
                vocab=129280, n_compressed=100000, prime_floor=1 << 19)


def is_prime(n: int) -> bool:
    if n < 2:
        return False
    if n % 2 == 0:
        return n == 2
    f = 3
    while f * f <= n:
        if n % f == 0:
            return False
        f += 2
    return True


def consecutive_primes(floor: int, count: int) -> list[int]:
    out, n = [], floor
    while len(out) < count:
        if is_prime(n):
            out.append(n)
        n += 1
    return out


@dataclasses.dataclass
class Tables:
    """Hash tables exactly as a loader would hand them over (consumed as given)."""

    token_map: np.ndarray    # int32 [vocab] -> compressed id
    pad_id: int              # compressed id used before a sequence starts
    multipliers: np.ndarray  # uint64 [max_ngram_size], one per look-back
    primes: np.ndarray       # uint64 [n_hash_cols]
    offsets: np.ndarray      # int64 [n_hash_cols], row offset of each slot in the table

    @property
    def num_embeddings(self) -> int:
        return int(self.offsets[-1]) + int(self.primes[-1])


def make_tables(geom: Geometry, rng: np.random.Generator, pad_id: int = 0) -> Tables:
    token_map = rng.integers(0, geom.n_compressed, size=geom.vocab, dtype=np.int32)
    multipliers = rng.integers(0, np.iinfo(np.uint64).max, size=geom.max_ngram_size,
                               dtype=np.uint64, endpoint=True) | np.uint64(1)
    primes = np.array(consecutive_primes(geom.prime_floor, geom.n_hash_cols), dtype=np.uint64)
    offsets = np.zeros(geom.n_hash_cols, dtype=np.int64)
    offsets[1:] = np.cumsum(primes[:-1].astype(np.int64))
    return Tables(token_map=token_map, pad_id=pad_id, multipliers=multipliers,
                  primes=primes, offsets=offsets)


@dataclasses.dataclass
class LayerHash:
    """One Engram layer's own hash constants and fp8 table, for calls that serve several layers.

    Each layer has its own entry of the hash layout (its own multipliers, primes, offsets and so
    its own number of table rows); the token map and pad id are shared (they live in Tables).
    table / scales are None when the caller draws them on the device instead.
    """

    multipliers: np.ndarray  # uint64 [max_ngram_size]
    primes: np.ndarray       # uint64 [n_hash_cols]
    offsets: np.ndarray      # int64 [n_hash_cols]
    table: np.ndarray | None
    scales: np.ndarray | None

    @property
    def num_embeddings(self) -> int:
        return int(self.offsets[-1]) + int(self.primes[-1])


def make_layer_hashes(geom: Geometry, n_layers: int, seed: int, prime_floor: int | None = None,
                      scale_mode: str = "pow2", with_tables: bool = True) -> list:
    """n_layers layers' hash constants (odd 64-bit multipliers; consecutive primes from a floor
    that grows by 1/8 per layer, so every layer's table has its own size; cumulative offsets) and,
    with_tables, their fp8 tables and e8m0 scales."""
    rng = np.random.default_rng(seed)
    floor = geom.prime_floor if prime_floor is None else prime_floor
    out = []
    for layer in range(n_layers):
        multipliers = rng.integers(0, np.iinfo(np.uint64).max, size=geom.max_ngram_size,
                                   dtype=np.uint64, endpoint=True) | np.uint64(1)
        primes = np.array(consecutive_primes(floor + layer * (floor // 8), geom.n_hash_cols),
                          dtype=np.uint64)
        offsets = np.zeros(geom.n_hash_cols, dtype=np.int64)
        offsets[1:] = np.cumsum(primes[:-1].astype(np.int64))
        rows = int(offsets[-1]) + int(primes[-1])
        table = make_fp8_rows(rows, geom.head_dim, rng) if with_tables else None
        scales = make_scales(rows, geom.head_dim, rng, scale_mode) if with_tables else None
        out.append(LayerHash(multipliers=multipliers, primes=primes, offsets=offsets,
                             table=table, scales=scales))
    return out


def make_fp8_rows_device(num_rows: int, head_dim: int, seed: int, device: str = "cuda"):
    """fp8 e4m3 codes [num_rows, head_dim] drawn on the device (torch generator): N(0,1) clamped
    to +-448, cast by torch. For workloads too large to draw on the host in time."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = torch.empty((num_rows, head_dim), dtype=torch.uint8, device=device)
    step = 1 << 22
    for r0 in range(0, num_rows, step):
        r1 = min(num_rows, r0 + step)
        v = torch.randn((r1 - r0, head_dim), generator=g, device=device).clamp_(-448.0, 448.0)
        out[r0:r1] = v.to(torch.float8_e4m3fn).view(torch.uint8)
    return out


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """bf16 storage bits of a float32 array (torch's round-to-nearest-even cast)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _no_zeros_bf16(bits: np.ndarray) -> np.ndarray:
    # Activations never hold +-0: a zero bf16 (probability ~0 for these draws) is nudged to the
    # smallest normal bf16 of the same sign, so "masked rows pass through bit-exactly" is not
    # muddied by the sign of zero.
    z = (bits & 0x7FFF) == 0
    if z.any():
        bits = bits.copy()
        bits[z] = (bits[z] & 0x8000) | 0x0080
    return bits


def make_fp8_rows(num_rows: int, head_dim: int, rng: np.random.Generator,
                  chunk_rows: int = 1 << 20) -> np.ndarray:
    """fp8 e4m3 codes [num_rows, head_dim]: N(0,1) clamped to +-448, cast by torch (RNE)."""
    out = np.empty((num_rows, head_dim), dtype=np.uint8)
    for r0 in range(0, num_rows, chunk_rows):
        r1 = min(num_rows, r0 + chunk_rows)
        v = rng.standard_normal((r1 - r0, head_dim), dtype=np.float32)
        np.clip(v, -448.0, 448.0, out=v)
        out[r0:r1] = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return out


def make_scales(num_rows: int, head_dim: int, rng: np.random.Generator | None,
                mode: str = "unit") -> np.ndarray:
    """e8m0 block scales [num_rows, head_dim/32]: 127 (= 1.0) or 127 + U{-4..4}."""
    nb = head_dim // SCALE_BLOCK
    if mode == "unit":
        return np.full((num_rows, nb), 127, dtype=np.uint8)
    if mode == "pow2":
        return (127 + rng.integers(-4, 5, size=(num_rows, nb))).astype(np.uint8)
    raise ValueError(mode)


def make_x(shape, rng: np.random.Generator, dist: str = "normal",
           chunk_elems: int = 1 << 24) -> np.ndarray:
    """bf16 residual streams x[..., hc, dim]: N(0,1), or Student-t(nu=3)/sqrt(3) (unit rms).

    Drawn in chunks of whole rows along the flattened leading axes, so large batches do not need
    float64 temporaries of their full size.
    """
    shape = tuple(shape)
    row = int(np.prod(shape[-2:]))
    rows = int(np.prod(shape[:-2])) if len(shape) > 2 else 1
    out = np.empty((rows, row), dtype=np.uint16)
    step = max(1, chunk_elems // row)
    for r0 in range(0, rows, step):
        n = min(step, rows - r0)
        if dist == "normal":
            v = rng.standard_normal((n, row), dtype=np.float32)
        elif dist == "student_t3":
            v = (rng.standard_t(3, size=(n, row)) / math.sqrt(3.0)).astype(np.float32)
        else:
            raise ValueError(dist)
        out[r0:r0 + n] = _no_zeros_bf16(f32_to_bf16_bits(v))
    return out.reshape(shape)


def make_x_device(shape, seed: int, dist: str = "normal", device: str = "cuda"):
    """Device-drawn x[..., hc, dim] as bf16 storage bits (torch int16), for benchmark batches too
    large to draw on the host in reasonable time: the distributions of make_x (N(0,1), or
    Student-t(nu=3)/sqrt(3) as a normal over sqrt(chi2_3 / 3)) from torch's generator seeded with
    `seed`, with the same nudge of exact zeros. The numbers differ from make_x's; parity tests use
    make_x."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    v = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if dist == "student_t3":
        # chi2 with 3 degrees of freedom as a sum of three squared normals
        c = torch.zeros_like(v)
        for _ in range(3):
            c.addcmul_(w := torch.randn(tuple(shape), generator=g, device=device), w)
        v = v / torch.sqrt(c / 3.0) / math.sqrt(3.0)
    elif dist != "normal":
        raise ValueError(dist)
    bits = v.to(torch.bfloat16).view(torch.int16)
    zero = (bits & 0x7FFF) == 0
    return torch.where(zero, (bits & -0x8000) | 0x0080, bits)


def make_wkv(geom: Geometry, rng: np.random.Generator) -> np.ndarray:
    """wkv weight [N, K] bf16: U(-1,1) * K^-0.5 (fixture rule scale = in^-0.5)."""
    v = rng.uniform(-1.0, 1.0, size=(geom.N, geom.K)).astype(np.float32)
    v *= np.float32(geom.K ** -0.5)
    return f32_to_bf16_bits(v)


def make_qk(geom: Geometry, rng: np.random.Generator) -> tuple[np.ndarray, np.ndarray]:
    """q_weight, k_weight [hc, dim] bf16: 1 + U(-0.05, 0.05) (fixture rule offset 1, +-0.05)."""
    q = 1.0 + rng.uniform(-0.05, 0.05, size=(geom.hc_mult, geom.dim))
    k = 1.0 + rng.uniform(-0.05, 0.05, size=(geom.hc_mult, geom.dim))
    return f32_to_bf16_bits(q.astype(np.float32)), f32_to_bf16_bits(k.astype(np.float32))


def make_tokens(geom: Geometry, B: int, T: int, rng: np.random.Generator) -> np.ndarray:
    return rng.integers(0, geom.vocab, size=(B, T), dtype=np.int32)


def make_span_mask(B: int, T: int, frac: float, rng: np.random.Generator,
                   mean_span: int = 256) -> np.ndarray:
    """bool [B, T]; False on seeded contiguous spans ("image positions") covering ~frac."""
    mask = np.ones((B, T), dtype=bool)
    for b in range(B):
        target = int(round(frac * T))
        covered = 0
        while covered < target:
            span = int(min(target - covered, max(1, rng.integers(mean_span // 2, 2 * mean_span))))
            start = int(rng.integers(0, max(1, T - span + 1)))
            before = int((~mask[b, start:start + span]).sum())
            mask[b, start:start + span] = False
            covered += span - before
    return mask


@dataclasses.dataclass
class Model:
    """One Engram layer's parameters and tables (all storage bits)."""

    geom: Geometry
    tables: Tables
    table: np.ndarray    # uint8 [num_embeddings, head_dim] e4m3 codes
    scales: np.ndarray   # uint8 [num_embeddings, head_dim/32] e8m0
    wkv: np.ndarray      # uint16 [N, K] bf16
    q: np.ndarray        # uint16 [hc, dim] bf16
    k: np.ndarray        # uint16 [hc, dim] bf16
    eps: float = 1e-6


def make_model(geom: Geometry, seed: int, scale_mode: str = "unit", pad_id: int = 0) -> Model:
    rng = np.random.default_rng(seed)
    tables = make_tables(geom, rng, pad_id=pad_id)
    rows = tables.num_embeddings
    table = make_fp8_rows(rows, geom.head_dim, rng)
    wkv = make_wkv(geom, rng)
    q, k = make_qk(geom, rng)
    # Scales are drawn last, so models that differ only in scale_mode share codes and weights.
    scales = make_scales(rows, geom.head_dim, rng, scale_mode)
    return Model(geom=geom, tables=tables, table=table, scales=scales, wkv=wkv, q=q, k=k)


@dataclasses.dataclass
class Batch:
    """One step's activations: tokens [B,T], x [B,T,hc,dim] bf16, token_mask [B,T] or None."""

    tokens: np.ndarray
    x: np.ndarray
    mask: np.ndarray | None


def make_batch(geom: Geometry, B: int, T: int, seed: int, x_dist: str = "normal",
               mask_frac: float = 0.0) -> Batch:
    rng = np.random.default_rng(seed)
    tokens = make_tokens(geom, B, T, rng)
    x = make_x((B, T, geom.hc_mult, geom.dim), rng, x_dist)
    mask = make_span_mask(B, T, mask_frac, rng) if mask_frac > 0 else None
    return Batch(tokens=tokens, x=x, mask=mask)


# Named workloads: (geometry, batch, tokens per sequence, extra knobs). The model of every full-width
# workload is drawn from the same seed, so they share tables and weights.
WORKLOADS = {
    "tiny": dict(geom=TINY, B=1, T=16, model_seed=BASE_SEED + 0, batch_seed=BASE_SEED + 100),
    "prefill_b1_t4096": dict(geom=FULL, B=1, T=4096, model_seed=BASE_SEED + 1,
                             batch_seed=BASE_SEED + 101),
    "decode_b64_ctx2048": dict(geom=FULL, B=64, T=1, prefill=2048, model_seed=BASE_SEED + 1,
                               batch_seed=BASE_SEED + 102),
    "masked_b8_t8192": dict(geom=FULL, B=8, T=8192, model_seed=BASE_SEED + 1,
                            batch_seed=BASE_SEED + 103, scale_mode="pow2",
                            x_dist="student_t3", mask_frac=0.10),
    "sweep_b1": dict(geom=FULL, B=1, T_list=(1, 8, 64, 512, 4096, 32768, 65536),
                     model_seed=BASE_SEED + 1, batch_seed=BASE_SEED + 104),
}
