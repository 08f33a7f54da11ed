"""Rotary position embedding applied at append time (oracle; test infrastructure only).

[Ch15 §15.3 硬件感知优化, "RoPE 与 Flash Attention 的融合"]: the rotation of
Q and K can be done in registers inside the kernel that already reads them,
instead of a separate pass through HBM; [FastGen §6] fuses it with the
blocked-KV write (linear_blocked_kv_rotary).  The pages defer RoPE's formula to
a section they do not include; the reading taken here is the rotate-half form:
for a head vector x of even length D at position p and i < D/2,

    x'[i]       = x[i] cos(p t_i) - x[i + D/2] sin(p t_i)
    x'[i + D/2] = x[i] sin(p t_i) + x[i + D/2] cos(p t_i)

with the caller's table of cos/sin values (the angles never enter here).  The
stored result is a decision of the cache dtype, so it is computed exactly as
the kernel does: in float32, every product and sum rounded on its own (no fused
multiply-add), then rounded to bf16 (nearest-even).  ``rotate_f64`` is the same
map in float64, used to pin the formula.
"""

import numpy as np


def rotate_f64(x, cos, sin):
    """x [..., D] float64; cos, sin [..., D/2] float64."""
    h = x.shape[-1] // 2
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * cos - x2 * sin, x1 * sin + x2 * cos], axis=-1)


def rotate_f32(x, cos, sin):
    """The kernel's arithmetic: float32, one rounding per product and per sum."""
    x = np.asarray(x, dtype=np.float32)
    cos = np.asarray(cos, dtype=np.float32)
    sin = np.asarray(sin, dtype=np.float32)
    h = x.shape[-1] // 2
    x1, x2 = x[..., :h], x[..., h:]
    a = x1 * cos
    b = x2 * sin
    c = x1 * sin
    d = x2 * cos
    return np.concatenate([a - b, c + d], axis=-1)


def f32_to_bf16_bits(x):
    """Round float32 to bf16 bit patterns, nearest-even (finite inputs)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    rounded = (u + 0x7FFF + lsb) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def rotate_storage(x, cos, sin, dtype):
    """Rotate values held in the storage dtype (float32, or bf16 bits) and store them back."""
    if dtype == "f32":
        return rotate_f32(x, cos, sin)
    return f32_to_bf16_bits(rotate_f32(bf16_bits_to_f32(x), cos, sin))


def append_rope(k_cache, v_cache, q, k, v, slot_mapping, positions, cos_sin, block_size, dtype,
                cache_append):
    """Rotate q and k at their positions, append rotated k and v, return rotated q.

    q [T, Hq, D] (or None), k, v [T, Hkv, D] in the storage dtype; cos_sin
    [max_position, D] float32 (cos of the D/2 angles, then their sin);
    ``cache_append`` is oracle.cache.append."""
    pos = np.asarray(positions)
    if np.any(pos < 0) or np.any(pos >= cos_sin.shape[0]):
        raise IndexError("position outside the table")
    h = k.shape[-1] // 2
    cos = cos_sin[pos][:, None, :h]
    sin = cos_sin[pos][:, None, h:]
    k_rot = rotate_storage(k, cos, sin, dtype)
    cache_append(k_cache, v_cache, k_rot, v, slot_mapping, block_size)
    return None if q is None else rotate_storage(q, cos, sin, dtype)


def rope_table(max_position, head_dim, base=10000.0):
    """cos/sin table [max_position, head_dim] (float32) with angles p * base^(-2i/D)."""
    h = head_dim // 2
    inv = base ** (-np.arange(h, dtype=np.float64) * 2.0 / head_dim)
    ang = np.arange(max_position, dtype=np.float64)[:, None] * inv[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)
