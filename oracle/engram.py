"""Oracle for the DeepSeek V4.1 Engram forward path: hash -> table rows -> wkv -> gate and add.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources, cited by page title and section:
  [listing]  page "DeepSeek V4.1" (blocks / engram-first / value), the Engram module listing
             (deepseek-ai/DeepSeek-V4.1-Flash inference/model.py, class Engram): __init__, forward.
  [gate]     page "DeepSeek V4.1 · Gate per stream": the formulas for a_k and g^e_k, the in/out
             shapes, and the parameter table (40,960 = 2 x 20,480).
  [docs]     page "Module engram" (deepseek_v41_ref engram, CPU reference): the four-stage list,
             the tables paragraph, structs EngramTables / NgramHashState and the function notes
             (e4m3_to_f32, embed_rows, f32_to_e4m3_rne, f32_to_e8m0_rne, gate_and_add,
             linear_bf16, regen_*).

Arrays cross this module as raw storage bits (bf16 -> uint16, fp8 -> uint8). All floating point is
float64; each function says where it rounds. Readings of the pages where they leave a step open
are marked "reading:".
"""
from __future__ import annotations

import numpy as np

from .numerics import bf16_to_f64, e4m3_to_f64, e8m0_to_f64, f64_to_bf16

GATE_CLAMP = 1e-6   # [listing] __init__: clamp_value; [gate] max(|a|, 10^-6)
SCALE_BLOCK = 32    # [docs] stage 2: one e8m0 scale per 32-element block


# ------------------------------------------------------------------------------ stage 1: hash


class NgramHashState:
    """Per-sequence look-back cache and n-gram hash ([docs] stage 1 and struct NgramHashState).

    The cache holds the compressed id of every position seen so far, so a later call (a decode
    step) looks back into what an earlier call (the prefill) pushed.

    Stage 1, in the order the docs give it:
      1. compressed token map: c_p = token_map[token_p];
      2. n-gram window with pad: the window of size n ending at position p holds c_{p-k},
         k = 0..n-1; a position before the sequence start holds ``pad_id``;
      3. per-look-back multiply: look-back k is multiplied by its own multiplier m_k;
      4. XOR-roll: mix_n = (c_p * m_0) XOR (c_{p-1} * m_1) XOR ... XOR (c_{p-n+1} * m_{n-1});
      5. % prime per (n-gram size, head), plus that slot's offset:
         id[s] = (mix_n mod P_s) + O_s,  s = (n - 2) * n_heads + head,  n = 2..max_ngram_size.

    Readings: multiply and XOR are on unsigned 64-bit words and wrap modulo 2^64; ``mod`` is the
    unsigned remainder; the multipliers are shared by all n and heads (so heads of one n differ only
    by their prime); slots are ordered n-major, then head, which is also the order of the
    flattened rows fed to wkv ([listing] forward: embed(hash_ids).flatten(-2)).
    """

    def __init__(self, token_map, pad_id, multipliers, primes, offsets, n_heads, max_ngram_size,
                 batch):
        self.token_map = np.asarray(token_map, dtype=np.int64)
        self.pad_id = int(pad_id)
        self.multipliers = np.asarray(multipliers, dtype=np.uint64)
        self.primes = np.asarray(primes, dtype=np.uint64)
        self.offsets = np.asarray(offsets, dtype=np.int64)
        self.n_heads = int(n_heads)
        self.max_ngram_size = int(max_ngram_size)
        self.cache = [np.zeros(0, dtype=np.int64) for _ in range(batch)]

    @property
    def n_hash_cols(self) -> int:
        return (self.max_ngram_size - 1) * self.n_heads

    def push(self, tokens: np.ndarray) -> np.ndarray:
        """Append tokens [B, T] to the caches; return hash ids [B, T, n_hash_cols] (int64)."""
        return self.push_layers(tokens, [(self.multipliers, self.primes, self.offsets)])[0]

    def push_layers(self, tokens: np.ndarray, layers) -> list:
        """Append tokens [B, T] to the caches once; return the hash ids of several Engram layers.

        ``layers`` holds one (multipliers, primes, offsets) per layer. Each Engram layer takes its
        own entry of the hash layout ([listing] __init__: layer_hash_index is the layer's place
        in layout.layer_ids, and its embedding has that entry's num_embeddings rows), so each
        layer has its own constants. Reading: the compressed token map and the cache of
        compressed ids depend only on the tokens, so one cache serves every layer; each layer's
        ids are formed from the same windows with its own constants. Returns a list with one
        int64 array [B, T, n_hash_cols] per layer.
        """
        tokens = np.asarray(tokens)
        B, T = tokens.shape
        outs = [np.empty((B, T, self.n_hash_cols), dtype=np.int64) for _ in layers]
        for b in range(B):
            p0 = len(self.cache[b])
            hist = np.concatenate([self.cache[b], self.token_map[tokens[b]]])   # step 1
            self.cache[b] = hist
            pos = p0 + np.arange(T)
            for out, (multipliers, primes, offsets) in zip(outs, layers):
                out[b] = self._slot_ids(hist, pos, np.asarray(multipliers, dtype=np.uint64),
                                        np.asarray(primes, dtype=np.uint64),
                                        np.asarray(offsets, dtype=np.int64))
        return outs

    def _slot_ids(self, hist, pos, multipliers, primes, offsets) -> np.ndarray:
        """Steps 2-5 for the positions ``pos`` of one sequence whose compressed ids are ``hist``."""
        out = np.empty((len(pos), self.n_hash_cols), dtype=np.int64)
        mix = np.zeros(len(pos), dtype=np.uint64)
        for n in range(1, self.max_ngram_size + 1):
            k = n - 1                                       # look-back of the new window cell
            q = pos - k
            c = np.where(q >= 0, hist[np.maximum(q, 0)], self.pad_id)      # step 2
            mix = mix ^ (c.astype(np.uint64) * multipliers[k])             # steps 3-4
            if n < 2:
                continue
            for head in range(self.n_heads):                                # step 5
                s = (n - 2) * self.n_heads + head
                out[:, s] = (mix % primes[s]).astype(np.int64) + offsets[s]
        return out


# ------------------------------------------------------------------------ stage 2: table rows


def embed_rows(table: np.ndarray, scales: np.ndarray, ids: np.ndarray) -> np.ndarray:
    """Gather rows by id and dequantise them ([docs] stage 2, functions embed_rows, regen_table).

    row[d] = e4m3(table[id, d]) * e8m0(scales[id, d // 32]), rounded to bf16. The product is
    exact in float64 (and in binary32), and e4m3 times a power of two is a bf16 value, so the
    rounding changes nothing within bf16's range. Returns bf16 bits [*ids.shape, head_dim].
    """
    ids = np.asarray(ids, dtype=np.int64)
    codes = table[ids]                                                   # [..., hd]
    sc = np.repeat(e8m0_to_f64(scales[ids]), SCALE_BLOCK, axis=-1)      # [..., hd]
    return f64_to_bf16(e4m3_to_f64(codes) * sc)


# ------------------------------------------------------------------------------- stage 3: wkv


def linear_bf16(a: np.ndarray, w: np.ndarray) -> np.ndarray:
    """kv = a @ w^T with a bf16 output ([docs] stage 3, function linear_bf16; [listing] wkv).

    a: bf16 bits [rows, in]; w: bf16 bits [out, in]; no bias. Reading of "f32 accumulate, bf16
    output": the exact sum, rounded once to bf16. Products of two bf16 values are exact in
    float64 and a float64 sum of at most a few thousand of them is within ~1e-13 (relative to the
    sum of magnitudes) of the exact value, so one rounding of it is the correctly rounded result
    except within that distance of a bf16 rounding boundary. Returns bf16 bits [rows, out].
    """
    A = bf16_to_f64(a)
    W = bf16_to_f64(w)
    return f64_to_bf16(A @ W.T)


# ---------------------------------------------------------------------- stage 4: gate and add


def gate_and_add(x: np.ndarray, kv: np.ndarray, q: np.ndarray, k: np.ndarray,
                 token_mask: np.ndarray | None, eps: float):
    """[listing] forward after the projection; [gate] a_k, g^e_k; [docs] function gate_and_add.

    x: bf16 bits [tokens, hc, dim]; kv: bf16 bits [tokens, dim * (hc + 1)]; q, k: bf16 bits
    [hc, dim]; token_mask: bool [tokens] or None (None = all True). Returns (out bf16 bits
    [tokens, hc, dim], gate float64 [tokens, hc]).

      key   = kv[:, :hc*dim] as [tokens, hc, dim];  value = kv[:, hc*dim:]     (the split)
      w     = q * k                                  (a product of two bf16: exact)
      rstd  = 1/sqrt(mean_d h^2 + eps) * 1/sqrt(mean_d key^2 + eps), per (token, stream)
      a     = (sum_d h * w * key) * rstd * dim^-1/2
      gate  = sigmoid(copysign(sqrt(max(|a|, 1e-6)), a));  gate = 0 where token_mask is False
      out   = bf16(h + gate * value), value shared by the hc streams

    Readings: the code's eps and copysign govern where the gate page's formula drops eps and
    writes sign(a) (so a = +0 gives sigmoid(+1e-3), not sigmoid(0)); the dot is a sum that starts
    from +0, so a dot whose terms are all -0 is +0. Everything is float64 and rounds once, at out.
    """
    x = np.asarray(x)
    M, hc, dim = x.shape
    h = bf16_to_f64(x)
    kvf = bf16_to_f64(np.asarray(kv).reshape(M, dim * (hc + 1)))
    key = kvf[:, : hc * dim].reshape(M, hc, dim)
    value = kvf[:, hc * dim:]
    w = bf16_to_f64(q) * bf16_to_f64(k)                                   # [hc, dim]
    rstd = 1.0 / np.sqrt((h * h).mean(-1) + eps) / np.sqrt((key * key).mean(-1) + eps)
    dot = 0.0 + (h * w[None] * key).sum(-1)
    a = dot * rstd * dim ** -0.5
    z = np.copysign(np.sqrt(np.maximum(np.abs(a), GATE_CLAMP)), a)
    gate = 1.0 / (1.0 + np.exp(-z))
    if token_mask is not None:
        gate = np.where(np.asarray(token_mask, dtype=bool)[:, None], gate, 0.0)
    out = f64_to_bf16(h + gate[:, :, None] * value[:, None, :])
    return out, gate


# -------------------------------------------------------------------------- the whole forward


def forward(state: NgramHashState, table, scales, wkv, q, k, x, tokens, token_mask, eps):
    """One Engram forward: hash the new tokens, gather rows, project, gate and add.

    x: bf16 bits [B, T, hc, dim]; tokens: [B, T]; token_mask: bool [B, T] or None.
    Returns a dict with hash_ids [B,T,24], rows [B,T,24,hd], kv [B,T,N], gate [B,T,hc] and out
    [B,T,hc,dim] (bits where the value is bf16).
    """
    B, T, hc, dim = x.shape
    hash_ids = state.push(tokens)
    rows = embed_rows(table, scales, hash_ids)                    # [B, T, 24, hd]
    a = rows.reshape(B * T, -1)                                   # flatten(-2)
    kv = linear_bf16(a, wkv)
    m = None if token_mask is None else np.asarray(token_mask).reshape(B * T)
    out, gate = gate_and_add(x.reshape(B * T, hc, dim), kv, q, k, m, eps)
    return dict(hash_ids=hash_ids, rows=rows, kv=kv.reshape(B, T, -1),
                gate=gate.reshape(B, T, hc), out=out.reshape(B, T, hc, dim))
