"""Vectorised float64 oracle of the Qwen3-style decoder forward with a KV cache.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain definitions in
numpy float64; no blocking, fusion or reordering beyond what the definitions
state.  numpy's matrix product is the only library primitive used.

Sources (page title, section):
* tinyllm L10.1 "Candle model runner ...", section 2.4 "The Llama forward,
  one step": RMSNorm with eps inside the square root, y = x W^T with weights
  stored [out, in], RoPE at the absolute position pos(t) = p_s + i, key j of a
  sequence stored at its absolute position, attention of token t over exactly
  the keys j <= pos(t) with scale 1/sqrt(D), x += o W_o^T, the SwiGLU MLP
  x += (silu(h2 W_g^T) * (h2 W_u^T)) W_d^T with h2 = RMSNorm(x), final norm
  and the tied LM head.
* octlm "A real model in our own decoder", section "Same design, bigger
  numbers, five switches": head_dim from the config (q/o projections are
  rectangular), ff_hidden from the config, rope_base 1e6, split-half RoPE
  (channel j pairs with j + D/2), and QK-norm (an RMSNorm on every query and
  key head before RoPE); section "Which channels rotate together" for the
  split-half pairing versus neighbour pairing.
* 1bit-MONSTER "Byte-identical", section "The rope table that was too
  accurate": phi = pos * 1e6^(-2j/128), evaluated here in float64.
* octlm "Proving it's the same model", section "Every logit, every position":
  logits at every position; the cached path splits the prompt in half.

Readings where the pages are silent:
* QK-norm gains have head_dim entries shared by all heads (this is what the
  published parameter count 596,049,920 requires).
* RoPE rotates like multiplication of (x_j + i x_{j+D/2}) by exp(i phi_j):
  out_j = x_j cos - x_{j+D/2} sin, out_{j+D/2} = x_{j+D/2} cos + x_j sin.
* Query head h reads key/value head floor(h * Hkv / H) (consecutive query
  heads share a key/value head).
* In the bf16 mode the oracle uses the bf16-rounded weights widened to
  float64; activations and the cache stay float64.
* In the int4 mode the seven projections of every layer are the int4
  effective weights (``oracle.int4``: groups of 32 input columns, f16
  scales) and the tied embedding is bf16-rounded; activations and the cache
  stay float64.

``mutant`` plants one named mistake (tinyllm L10.1 section 5 "Pitfalls",
and octlm's neighbour pairing) so that tests can show the parity harness
detects it.  The product never sets it.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import int4
from .numerics import bf16_round

MUTANTS = ("s13", "s14", "s15", "s16", "s20", "s22", "neighbour")


@dataclass(frozen=True)
class DecoderConfig:
    vocab: int
    d_model: int
    n_layers: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ff_hidden: int
    rope_base: float = 1e6
    rms_eps: float = 1e-6
    max_positions: int = 4096
    block_tokens: int = 16


def param_count(cfg: DecoderConfig) -> int:
    """Unique parameters of the tied-embedding decoder."""
    d, H, Hkv, D, F = cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ff_hidden
    per_layer = (
        d  # attention RMSNorm gain
        + H * D * d + 2 * Hkv * D * d  # W_q, W_k, W_v
        + 2 * D  # q_norm, k_norm gains (shared by heads)
        + d * H * D  # W_o
        + d  # MLP RMSNorm gain
        + 3 * F * d  # W_gate, W_up, W_down
    )
    return cfg.vocab * d + cfg.n_layers * per_layer + d


def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * w over the last axis."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * w


def rope_angles(pos: np.ndarray, head_dim: int, base: float, reverse: bool = False) -> np.ndarray:
    """phi[t, j] = pos_t * base^(-2j/D), j = 0 .. D/2-1, in float64."""
    j = np.arange(head_dim // 2, dtype=np.float64)
    if reverse:  # mutant s20: frequencies in reversed order
        j = j[::-1]
    theta = base ** (-2.0 * j / head_dim)
    return np.asarray(pos, dtype=np.float64)[:, None] * theta[None, :]


def rope(x: np.ndarray, pos: np.ndarray, base: float, split: bool = True, reverse: bool = False) -> np.ndarray:
    """Rotate x[t, ..., D] by the angles of position pos[t].

    split=True pairs channel j with j + D/2 (Qwen); split=False pairs 2j with
    2j+1 (the neighbour layout, a valid RoPE but not Qwen's).
    """
    D = x.shape[-1]
    phi = rope_angles(pos, D, base, reverse)
    extra = x.ndim - 2
    phi = phi.reshape(phi.shape[:1] + (1,) * extra + phi.shape[1:])
    c, s = np.cos(phi), np.sin(phi)
    if split:
        a, b = x[..., : D // 2], x[..., D // 2:]
        return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)
    a, b = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = b * c + a * s
    return out


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def attention_one(q: np.ndarray, keys: np.ndarray, values: np.ndarray) -> np.ndarray:
    """softmax(q . k_j / sqrt(D)) weighted sum of v_j over the given keys.

    q [D], keys [n, D], values [n, D]."""
    s = keys @ q / np.sqrt(q.shape[-1])
    p = np.exp(s - s.max())
    p /= p.sum()
    return p @ values


@dataclass
class SeqCache:
    """Per-sequence float64 cache: k[l][pos, kv_head, D], v likewise."""
    k: list
    v: list
    length: int = 0  # positions written so far (highest written + 1)
    written: list = field(default_factory=list)


class Oracle:
    """The decoder of the pages, evaluated in float64.

    weights: dict name -> float32 (or float64) array, names as in
    ``decoder_qwen3_step_gb300.inputs.weight_names``.  mode "fp32" widens
    the weights as given; mode "bf16" first rounds every matrix (embedding
    included) to bfloat16, keeping the RMSNorm gains as given; mode "int4"
    quantizes the projections (q, k, v, o, gate, up, down) to int4 with
    f16 group scales and rounds the embedding to bfloat16.
    """

    def __init__(self, cfg: DecoderConfig, weights: dict, mode: str = "fp32"):
        if mode not in ("fp32", "bf16", "int4"):
            raise ValueError(mode)
        if cfg.n_heads % cfg.n_kv_heads or cfg.head_dim % 2:
            raise ValueError("n_heads must be a multiple of n_kv_heads and head_dim even")
        self.cfg = cfg
        self.mode = mode

        def mat(name):
            w = np.asarray(weights[name], dtype=np.float32)
            if mode == "int4" and name != "embed":
                return int4.effective(w)
            if mode in ("bf16", "int4"):
                w = bf16_round(w)
            return w.astype(np.float64)

        def gain(name):
            return np.asarray(weights[name], dtype=np.float64)

        self.embed = mat("embed")
        self.final_norm = gain("final_norm")
        self.layers = []
        for l in range(cfg.n_layers):
            p = f"layers.{l}."
            self.layers.append({
                "attn_norm": gain(p + "attn_norm"),
                "q": mat(p + "q"), "k": mat(p + "k"), "v": mat(p + "v"),
                "q_norm": gain(p + "q_norm"), "k_norm": gain(p + "k_norm"),
                "o": mat(p + "o"),
                "mlp_norm": gain(p + "mlp_norm"),
                "gate": mat(p + "gate"), "up": mat(p + "up"), "down": mat(p + "down"),
            })

    # -- cache --------------------------------------------------------------
    def new_cache(self, max_positions: int | None = None) -> SeqCache:
        cfg = self.cfg
        n = max_positions or cfg.max_positions
        shape = (n, cfg.n_kv_heads, cfg.head_dim)
        return SeqCache(k=[np.zeros(shape) for _ in range(cfg.n_layers)],
                        v=[np.zeros(shape) for _ in range(cfg.n_layers)],
                        written=[np.zeros(n, dtype=bool) for _ in range(cfg.n_layers)])

    # -- one step of one sequence ---------------------------------------------
    def forward(self, cache: SeqCache, tokens, start: int, rows: str = "all",
                mutant: str | None = None, dump: list | None = None) -> np.ndarray:
        """Run the new tokens tokens[0..n) at positions start..start+n-1.

        Writes their K/V into ``cache`` and returns float64 logits: one row
        per new token (rows="all") or only the last one (rows="last").
        ``dump``, when given, receives the residual stream after the
        embedding and after every layer.
        """
        cfg = self.cfg
        if mutant is not None and mutant not in MUTANTS:
            raise ValueError(mutant)
        tokens = np.asarray(tokens, dtype=np.int64)
        n = tokens.shape[0]
        if n == 0:
            raise ValueError("empty step")
        if np.any(tokens < 0) or np.any(tokens >= cfg.vocab):
            raise ValueError("token id outside the vocabulary")
        pos = start + np.arange(n)
        if pos[-1] >= cache.k[0].shape[0]:
            raise ValueError("position past the cache")
        H, Hkv, D = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
        rope_pos = np.arange(n) if mutant == "s13" else pos
        split = mutant != "neighbour"
        reverse = mutant == "s20"

        x = self.embed[tokens].copy()
        if dump is not None:
            dump.append(x.copy())
        for l, w in enumerate(self.layers):
            h = rms_norm(x, w["attn_norm"], cfg.rms_eps)
            q = (h @ w["q"].T).reshape(n, H, D)
            k = (h @ w["k"].T).reshape(n, Hkv, D)
            v = (h @ w["v"].T).reshape(n, Hkv, D)
            q = rms_norm(q, w["q_norm"], cfg.rms_eps)
            k = rms_norm(k, w["k_norm"], cfg.rms_eps)
            q = rope(q, rope_pos, cfg.rope_base, split, reverse)
            k = rope(k, rope_pos, cfg.rope_base, split, reverse)
            cache.k[l][pos] = k
            cache.v[l][pos] = k if mutant == "s15" else v
            cache.written[l][pos] = True

            o = np.empty((n, H, D))
            G = H // Hkv
            for t in range(n):
                last = t if mutant == "s14" else pos[t]  # s14: q_offset 0
                if not cache.written[l][: last + 1].all():
                    raise ValueError("attention reads a position that was never written")
                keys = cache.k[l][: last + 1]  # [P, Hkv, D]
                vals = cache.v[l][: last + 1]
                # query head h = g*G + i reads key/value head g = floor(h*Hkv/H)
                qg = q[t].reshape(Hkv, G, D)
                s = np.matmul(qg, keys.transpose(1, 2, 0)) / np.sqrt(D)  # [Hkv, G, P]
                p = np.exp(s - s.max(axis=-1, keepdims=True))
                p /= p.sum(axis=-1, keepdims=True)
                o[t] = np.matmul(p, vals.transpose(1, 0, 2)).reshape(H, D)
            x = x + o.reshape(n, H * D) @ w["o"].T

            h2 = rms_norm(x, w["mlp_norm"], cfg.rms_eps)
            g_ = h2 @ w["gate"].T
            u_ = h2 @ w["up"].T
            act = silu(u_) * g_ if mutant == "s22" else silu(g_) * u_
            x = x + act @ w["down"].T
            if dump is not None:
                dump.append(x.copy())

        cache.length = max(cache.length, int(pos[-1]) + 1)
        if rows == "last":
            x = x[-1:]
        elif rows != "all":
            raise ValueError(rows)
        hf = x if mutant == "s16" else rms_norm(x, self.final_norm, cfg.rms_eps)
        return hf @ self.embed.T

    # -- paths ----------------------------------------------------------------
    def full(self, tokens, mutant=None) -> np.ndarray:
        """The whole prompt in one step; logits at every position."""
        return self.forward(self.new_cache(len(tokens) + 1), tokens, 0, mutant=mutant)

    def cached(self, tokens, mutant=None) -> np.ndarray:
        """First half, then the second half on top of the first half's cache."""
        split = max(1, len(tokens) // 2)
        cache = self.new_cache(len(tokens) + 1)
        a = self.forward(cache, tokens[:split], 0, mutant=mutant)
        if split == len(tokens):
            return a
        b = self.forward(cache, tokens[split:], split, mutant=mutant)
        return np.concatenate([a, b], axis=0)

    def greedy(self, cache: SeqCache, first_id: int, start: int, steps: int, mutant=None):
        """Greedy decode: feed one token per step; return (ids fed, logits)."""
        ids, rows = [], []
        tok = int(first_id)
        for i in range(steps):
            logits = self.forward(cache, [tok], start + i, mutant=mutant)[0]
            ids.append(tok)
            rows.append(logits)
            tok = int(np.argmax(logits))  # first maximum = lowest id on ties
        return ids, np.stack(rows)


def argmax_lowest(logits: np.ndarray) -> np.ndarray:
    """Greedy ids, ties to the lowest id (numpy returns the first maximum)."""
    return np.argmax(logits, axis=-1)
