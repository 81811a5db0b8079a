"""Counter-based activations and weights (inputs only; no arithmetic of the method).

A token's values come from numpy's Philox counter generator keyed by
``(path key, stream)``.  The path key folds the token ids along the token's
root path, so the same logical token (same content prefix, same question prefix)
gets the same values wherever it is packed, alone or among thousands of other
inputs, and a floor question gets the same values as a user input holding that
question on empty content.

Values are drawn in fp32 and rounded to bf16 (round-to-nearest-even) by torch.
"""
from __future__ import annotations

import numpy as np
import torch

MASK = (1 << 64) - 1
STREAM_Q, STREAM_K, STREAM_V, STREAM_H = 1, 2, 3, 4


def _mix(a: int, b: int) -> int:
    """splitmix64 finaliser of ``a ^ golden * (b + 1)``."""
    z = (a ^ ((0x9E3779B97F4A7C15 * (b + 1)) & MASK)) & MASK
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK
    return z ^ (z >> 31)


def root_key(seed: int) -> int:
    return _mix(0x5EED0000 + seed, 0)


def path_keys(tok, parent, T, seed=0):
    """Key of every row ``< T`` of a packed layout from its token id and its parent row."""
    keys = [0] * T
    r0 = root_key(seed)
    for r in range(T):
        p = int(parent[r])
        keys[r] = _mix(keys[p] if p >= 0 else r0, int(tok[r]))
    return keys


def seq_keys(tokens, seed=0):
    """Keys of a plain (unpacked) token sequence: row ``i``'s parent is ``i - 1``."""
    keys, k = [], root_key(seed)
    for t in tokens:
        k = _mix(k, int(t))
        keys.append(k)
    return keys


def extend_key(key, token):
    """Key of a row whose token ``token`` follows the row with key ``key`` on a root path
    (a decoded token appended to a searched slot's path)."""
    return _mix(int(key), int(token))


def normal_rows(keys, stream, n):
    """``[len(keys), n]`` fp32 N(0, 1) values, one Philox stream per distinct key."""
    out = np.empty((len(keys), n), dtype=np.float32)
    cache = {}
    for i, k in enumerate(keys):
        row = cache.get(k)
        if row is None:
            g = np.random.Generator(np.random.Philox(key=np.array([k, stream], dtype=np.uint64)))
            row = g.standard_normal(n, dtype=np.float32)
            cache[k] = row
        out[i] = row
    return out


def bf16(x):
    """Round an fp32 array to a bf16 torch tensor (nearest-even)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def qkv(keys, T_pad, n_q_heads, n_kv_heads, d_head):
    """Packed bf16 ``q [T_pad, Hq, d]``, ``k``, ``v [T_pad, Hkv, d]``; pad rows are zero."""
    T = len(keys)

    def make(stream, H):
        a = np.zeros((T_pad, H * d_head), dtype=np.float32)
        a[:T] = normal_rows(keys, stream, H * d_head)
        return bf16(a).reshape(T_pad, H, d_head)

    return make(STREAM_Q, n_q_heads), make(STREAM_K, n_kv_heads), make(STREAM_V, n_kv_heads)


def hidden(keys, T_pad, d_model, rows=None):
    """Packed bf16 final hidden states ``[T_pad, D]``; only ``rows`` (default all) are drawn."""
    a = np.zeros((T_pad, d_model), dtype=np.float32)
    rows = range(len(keys)) if rows is None else rows
    rows = np.asarray(list(rows), dtype=np.int64)
    if len(rows):
        a[rows] = normal_rows([keys[r] for r in rows], STREAM_H, d_model)
    return bf16(a)


def lm_head(vocab, d_model, seed=0, device="cpu"):
    """bf16 lm-head ``[V, D]`` with entries N(0, 1/D).

    On the CPU it is drawn by numpy's Philox (reproducible everywhere); on a CUDA
    device by torch's seeded generator (fast, reproducible for one torch build).
    """
    std = 1.0 / np.sqrt(d_model)
    if str(device).startswith("cuda"):
        g = torch.Generator(device=device)
        g.manual_seed(0x1E4D + seed)
        w = torch.empty((vocab, d_model), dtype=torch.float32, device=device)
        out = torch.empty((vocab, d_model), dtype=torch.bfloat16, device=device)
        step = max(1, (1 << 26) // d_model)
        for v0 in range(0, vocab, step):
            v1 = min(vocab, v0 + step)
            w[:v1 - v0].normal_(0.0, std, generator=g)
            out[v0:v1] = w[:v1 - v0].to(torch.bfloat16)
        return out
    g = np.random.Generator(np.random.Philox(key=np.array([0x1E4D + seed, 7], dtype=np.uint64)))
    return bf16(g.standard_normal((vocab, d_model), dtype=np.float32) * np.float32(std))


def e4m3_rows(w_bf16):
    """Per-row e4m3 weights for an lm-head: ``(codes uint8 [V, D], scale fp32 [V])``.

    ``scale = absmax / 448`` per row; codes are torch's saturating-free cast of
    the clamped quotient (round-to-nearest-even).  Works on CPU or CUDA tensors.
    """
    w = w_bf16.float()
    absmax = w.abs().amax(dim=1)
    scale = torch.where(absmax == 0, torch.ones_like(absmax), absmax / 448.0)
    q = (w / scale[:, None]).clamp_(-448.0, 448.0)
    codes = q.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale.contiguous()
