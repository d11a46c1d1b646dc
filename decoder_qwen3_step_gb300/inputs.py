"""Seeded synthetic inputs: decoder shapes, random-init weights and token ids.

This module holds no arithmetic of the decoder itself.  It is the one place
shared by the CUDA path, the tests and the float64 oracle, so both sides are
fed the very same arrays.

Shapes and recipes:
* "tiny": vocab 512, d_model 64, 2 layers, 4 query / 2 key-value heads,
  head_dim 32, ff_hidden 192; one 16-token prompt.
* "small": vocab 8192, d_model 512, 8 layers, 8 / 4 heads, head_dim 64,
  ff_hidden 1536; 4 prompts of 128 tokens.
* "qwen3_0p6b": the Qwen3-0.6B shape (octlm "A real model in our own
  decoder": vocab 151,936, d_model 1,024, 28 layers, 16 query heads of 128,
  8 key-value heads, ff_hidden 3,072, rope_base 1e6, rms_norm_eps 1e-6),
  596,049,920 parameters.

Weights are N(0, 0.02) float32 drawn from numpy's PCG64 seeded with 0, one
tensor at a time in ``weight_names`` order; RMSNorm gains are 1.  Token ids
are uniform on [0, vocab) from PCG64 seeded with 1.
"""

from __future__ import annotations

import numpy as np

SHAPES = {
    "tiny": dict(vocab=512, d_model=64, n_layers=2, n_heads=4, n_kv_heads=2, head_dim=32, ff_hidden=192),
    "small": dict(vocab=8192, d_model=512, n_layers=8, n_heads=8, n_kv_heads=4, head_dim=64, ff_hidden=1536),
    "qwen3_0p6b": dict(vocab=151936, d_model=1024, n_layers=28, n_heads=16, n_kv_heads=8, head_dim=128,
                       ff_hidden=3072),
}
ROPE_BASE = 1e6
RMS_EPS = 1e-6
BLOCK_TOKENS = 16

LAYER_TENSORS = ("attn_norm", "q", "k", "v", "q_norm", "k_norm", "o", "mlp_norm", "gate", "up", "down")


def weight_names(shape: dict) -> list[str]:
    names = ["embed"]
    for l in range(shape["n_layers"]):
        names += [f"layers.{l}.{t}" for t in LAYER_TENSORS]
    return names + ["final_norm"]


def weight_shape(shape: dict, name: str) -> tuple:
    d, H, Hkv, D, F, V = (shape[k] for k in ("d_model", "n_heads", "n_kv_heads", "head_dim", "ff_hidden", "vocab"))
    leaf = name.rsplit(".", 1)[-1]
    return {
        "embed": (V, d), "final_norm": (d,), "attn_norm": (d,), "mlp_norm": (d,),
        "q": (H * D, d), "k": (Hkv * D, d), "v": (Hkv * D, d), "q_norm": (D,), "k_norm": (D,),
        "o": (d, H * D), "gate": (F, d), "up": (F, d), "down": (d, F),
    }[leaf]


def make_weights(shape: dict, seed: int = 0, std: float = 0.02) -> dict:
    """Random-init float32 weights; norm gains are ones."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = {}
    for name in weight_names(shape):
        shp = weight_shape(shape, name)
        if name.endswith("norm"):
            out[name] = np.ones(shp, dtype=np.float32)
        else:
            a = rng.standard_normal(shp, dtype=np.float32)
            a *= np.float32(std)
            out[name] = a
    return out


def make_ids(vocab: int, count: int, seed: int = 1) -> np.ndarray:
    """Uniform token ids on [0, vocab) as int32."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.integers(0, vocab, size=count, dtype=np.int64).astype(np.int32)


def serving_context_lengths(n_seqs: int = 32, lo: int = 1024, hi: int = 2048) -> list[int]:
    """Distinct context lengths lo..hi spread evenly over n_seqs sequences.

    Sequence s keeps the first lo + round(s * (hi - lo) / (n_seqs - 1)) of
    its 2,048 preloaded ids (1024 ... 2048 for 32 sequences)."""
    if n_seqs == 1:
        return [hi]
    return [lo + int(round(s * (hi - lo) / (n_seqs - 1))) for s in range(n_seqs)]
