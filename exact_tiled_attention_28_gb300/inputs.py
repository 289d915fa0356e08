"""Seeded synthetic inputs for exact attention.

Both sides of every parity check draw from this module: the CUDA path (through
the Python binding) and the fp64 oracle. It holds none of the attention
arithmetic, only random numbers and the bf16 storage format.

Recipe (the workloads of the pages draw Q, K, V and dO i.i.d. N(0, 1) and run
them in bf16):

* one independent stream per (seed, tensor, batch index, head index): a
  Philox-4x64 counter generator keyed by those four numbers, so any single
  head can be regenerated without drawing the others;
* ``standard_normal`` in float32 from that stream, shape [N, d];
* rounded to bf16 with round-to-nearest-even on the float32 bit pattern.

The bf16 values are returned as their raw ``uint16`` bit patterns. The CUDA
path takes those bits as-is; the oracle widens them exactly to float64 with
:func:`bf16_bits_to_f64`.
"""

from __future__ import annotations

import numpy as np

TENSOR_IDS = {"q": 0, "k": 1, "v": 2, "do": 3}


def _philox_key(seed: int, tensor: str, b: int, h: int) -> int:
    tid = TENSOR_IDS[tensor]
    if not (0 <= seed < 2**32 and 0 <= b < 2**24 and 0 <= h < 2**24):
        raise ValueError("seed, batch or head index out of range")
    return (seed << 64) | (tid << 48) | (b << 24) | h


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even).

    Returns the 16-bit patterns as ``uint16``. Inputs must be finite.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 exactly."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float64 exactly."""
    return bf16_bits_to_f32(bits).astype(np.float64)


def head_bits(seed: int, tensor: str, b: int, h: int, N: int, d: int) -> np.ndarray:
    """bf16 bits [N, d] of one head of one tensor."""
    rng = np.random.Generator(np.random.Philox(key=_philox_key(seed, tensor, b, h)))
    return f32_to_bf16_bits(rng.standard_normal((N, d), dtype=np.float32))


def tensor_bits(seed: int, tensor: str, B: int, H: int, N: int, d: int) -> np.ndarray:
    """bf16 bits [B, H, N, d] of a whole tensor (row-major, d innermost)."""
    out = np.empty((B, H, N, d), dtype=np.uint16)
    for b in range(B):
        for h in range(H):
            out[b, h] = head_bits(seed, tensor, b, h, N, d)
    return out


def attention_inputs(seed: int, B: int, H: int, N: int, d: int,
                     tensors=("q", "k", "v", "do")) -> dict:
    """Dict tensor name -> bf16 bits [B, H, N, d]."""
    return {t: tensor_bits(seed, t, B, H, N, d) for t in tensors}


# Inputs of unequal lengths: q and dO of (sequence b, head h) come from
# ``seed``, k and v from ``seed + KV_SEED_OFFSET``, each block drawn for its own
# length.
KV_SEED_OFFSET = 500


def nqnk_inputs(seed: int, B: int, H: int, Nq: int, Nk: int, d: int) -> dict:
    """Dict name -> bf16 bits: q, do [B, H, Nq, d] and k, v [B, H, Nk, d]."""
    out = attention_inputs(seed, B, H, Nq, d, ("q", "do"))
    out.update(attention_inputs(seed + KV_SEED_OFFSET, B, H, Nk, d, ("k", "v")))
    return out


def packed_inputs(seed: int, lens_q, lens_k, H: int, d: int):
    """A packed batch: (dict name -> bf16 bits [T, H, d] with q, do on
    sum(lens_q) rows and k, v on sum(lens_k) rows, cu_q, cu_k int32 prefix
    offsets). Block (b, h) of each tensor is the head generator's [n, d] draw."""
    cu_q = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    out = {n: np.zeros((int(cu[-1]), H, d), dtype=np.uint16)
           for n, cu in (("q", cu_q), ("do", cu_q), ("k", cu_k), ("v", cu_k))}
    for b, (nq, nk) in enumerate(zip(lens_q, lens_k)):
        for h in range(H):
            for n, s, cu, length in (("q", seed, cu_q, nq), ("do", seed, cu_q, nq),
                                     ("k", seed + KV_SEED_OFFSET, cu_k, nk),
                                     ("v", seed + KV_SEED_OFFSET, cu_k, nk)):
                out[n][cu[b]:cu[b + 1], h] = head_bits(s, n, b, h, int(length), d)
    return out, cu_q, cu_k


def head_inputs_f64(seed: int, b: int, h: int, N: int, d: int,
                    tensors=("q", "k", "v", "do")) -> dict:
    """Dict tensor name -> float64 [N, d] for one head (exact bf16 values)."""
    return {t: bf16_bits_to_f64(head_bits(seed, t, b, h, N, d)) for t in tensors}


def bits_to_torch_bf16(bits: np.ndarray):
    """View bf16 bit patterns as a CPU ``torch.bfloat16`` tensor (no copy of values)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def torch_bf16_to_bits(t) -> np.ndarray:
    """Raw bf16 bit patterns of a ``torch.bfloat16`` tensor, moved to the host."""
    import torch
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
