"""Each PEFT method computed from its own definition (float64, row vectors).

Test infrastructure only (see ``oracle/__init__``).

Orientation follows the article's normal-form equation, which writes ``xW``:
x is [n, d_in], W is [d_in, d_out]; a "column" is an output feature.
"""
from __future__ import annotations

import numpy as np


def base(x: np.ndarray, W: np.ndarray) -> np.ndarray:
    """No adapter: the shared GEMM ``h = xW`` (article, "The big picture",
    description of batched LoRA serving)."""
    return x @ W


def lora(x, W, A, B, c):
    """LoRA: ``y = x (W + c A B)`` with c the scalar of the low-rank term
    (article, "The big picture": a low-rank term A, B with scalar c)."""
    return x @ (W + c * (A @ B))


def dora_scale(W, A, B, c, m):
    """DoRA's per-column factor: learned length m over the L2 norm of each
    column of ``W + cAB`` (article, "How does Scute plug into vLLM?": s is the
    learned length divided by the norm of each column of W+cAB)."""
    Wp = W + c * (A @ B)
    norms = np.sqrt(np.sum(Wp * Wp, axis=0))
    return m / norms


def dora(x, W, A, B, c, m):
    """DoRA: rescale every column of ``W' = W + cAB`` to the learned length m,
    ``y = x W' diag(m / ||col W'||)`` (article, "What problem is it solving?":
    DoRA rescales each output column to a learned length)."""
    Wp = W + c * (A @ B)
    norms = np.sqrt(np.sum(Wp * Wp, axis=0))
    return x @ (Wp * (m / norms)[None, :])


def ia3(x, W, l):
    """(IA)^3 on a key, value or up projection: ``y = (xW) * l`` (article,
    "What problem is it solving?" and "The big picture": l multiplies the
    keys, the values and, after reordering, the up projection's output)."""
    return (x @ W) * l


def silu(z):
    return z / (1.0 + np.exp(-z))


def ia3_ffn(x, Wg, Wu, l, act=silu):
    """(IA)^3 on the FFN intermediate as defined: ``act(x Wg) * (x Wu) * l``."""
    return act(x @ Wg) * (x @ Wu) * l


def ia3_ffn_reordered(x, Wg, Wu, l, act=silu):
    """The reordering the article uses to make l the s slot of the up
    projection: ``act(x Wg) * ((x Wu) * l)`` ("The big picture")."""
    return act(x @ Wg) * ((x @ Wu) * l)


def vera(x, W, A_sh, B_sh, d, e):
    """VeRA: shared frozen A, B; per-adapter d between them and e after B,
    ``y = xW + ((x A_sh) * d) B_sh * e`` (article, "The big picture": VeRA's
    two vectors are d and e; "Which slots can be merged at load?")."""
    return x @ W + (((x @ A_sh) * d) @ B_sh) * e


def block_diag(blocks: np.ndarray) -> np.ndarray:
    """Assemble the block-diagonal matrix from blocks [n_blk, b, b]; block k
    acts on input features [k b, (k+1) b)."""
    nb, b, _ = blocks.shape
    R = np.zeros((nb * b, nb * b), dtype=np.float64)
    for k in range(nb):
        R[k * b:(k + 1) * b, k * b:(k + 1) * b] = blocks[k]
    return R


def oft(x, W, R_blocks):
    """OFT: multiply the layer input by the block-diagonal rotation,
    ``y = (x R) W`` (article, "What problem is it solving?": OFT multiplies each
    layer's input by a block-diagonal rotation matrix)."""
    return (x @ block_diag(R_blocks)) @ W
