"""Helpers shared by the GPU parity tests (no layer arithmetic here)."""
import numpy as np


def to_dev_bf16(bits, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def bf16_bits_of(t):
    """torch bf16 tensor -> numpy uint16 bit patterns."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f64(t):
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def max_abs_rel(got, want):
    """max_i |got_i - want_i| / max_i |want_i| (the tolerance metric of the layer)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    den = np.abs(want).max()
    if den == 0:
        return float(np.abs(got).max())
    return float(np.abs(got - want).max() / den)


def near_tie_tokens(logits, k, gap):
    """Tokens whose k-th and (k+1)-th largest logits are within `gap`."""
    L = np.sort(np.asarray(logits, dtype=np.float64), axis=1)[:, ::-1]
    if L.shape[1] <= k:
        return np.zeros(L.shape[0], dtype=bool)
    return (L[:, k - 1] - L[:, k]) < gap


def sf_index(rows, kblocks):
    """Byte offset of the scale of (row r, K-block b) in the MOE_SF layout that
    include/moe.h documents (a pure index permutation)."""
    r = np.arange(rows)[:, None]
    b = np.arange(kblocks)[None, :]
    return (((r // 128) * (kblocks // 4) + b // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4
            + (b % 4))


def sf_pack(scales):
    """Row-major scales [rows, K/32] -> flat MOE_SF buffer."""
    rows, kb = scales.shape
    buf = np.zeros(rows * kb, dtype=np.uint8)
    buf[sf_index(rows, kb)] = scales
    return buf


def sf_unpack(buf, rows, kblocks):
    """Flat MOE_SF buffer -> row-major scales [rows, K/32]."""
    return np.asarray(buf).reshape(-1)[: rows * kblocks][sf_index(rows, kblocks)]
