"""Pins for the 8-bit KV oracle (CPU only)."""

import numpy as np

from oracle import attention, numerics, quant


def _bf16(x):
    import torch

    t = torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_error_is_at_most_half_a_step():
    rng = np.random.default_rng(0)
    x = _bf16(rng.standard_normal((50, 4, 128)) * 3)
    codes, scale = quant.quantize_rows(x, "bf16")
    back = quant.dequantize(codes, scale)
    f = numerics.widen(x, "bf16")
    step = scale.astype(np.float64)[..., None]
    # half a step, plus the float32 rounding of x / scale (|x / scale| <= 127, one
    # rounding of 2^-24 relative) and of the scale itself
    assert np.all(np.abs(back - f) <= step * (0.5 + 127 * 2.0 ** -23))
    # the largest magnitude of each row maps to +-127
    assert np.all(np.max(np.abs(codes.astype(int)), axis=-1) == 127)


def test_symmetric_zero_row_and_exact_grid():
    x = np.zeros((1, 1, 64), np.float32)
    x[0, 0, 3] = 127.0
    x[0, 0, 7] = -5.0
    c, s = quant.quantize_rows(x, "f32")
    assert s[0, 0] == 1.0 and c[0, 0, 3] == 127 and c[0, 0, 7] == -5   # values on the grid
    c2, s2 = quant.quantize_rows(-x, "f32")
    assert np.array_equal(c2, -c) and np.array_equal(s2, s)
    cz, sz = quant.quantize_rows(np.zeros((2, 3, 64), np.float32), "f32")
    assert np.all(cz == 0) and np.all(sz == 0)
    # ties go to the even code: 2.5 and 3.5 steps
    y = np.zeros((1, 1, 64), np.float32)
    y[0, 0, 0] = 127.0
    y[0, 0, 1] = 2.5
    y[0, 0, 2] = 3.5
    cy, _ = quant.quantize_rows(y, "f32")
    assert cy[0, 0, 1] == 2 and cy[0, 0, 2] == 4


def test_int8_decode_equals_exact_attention_on_dequantised_values():
    rng = np.random.default_rng(1)
    hkv, d, bs = 2, 32, 4
    nb = 10
    k = _bf16(rng.standard_normal((20, hkv, d)))
    v = _bf16(rng.standard_normal((20, hkv, d)))
    kq = np.zeros((nb, hkv, bs, d), np.int8)
    vq = np.zeros_like(kq)
    ks = np.zeros((nb, hkv, bs), np.float32)
    vs = np.zeros_like(ks)
    slots = np.arange(20) + 8                                  # blocks 2..6
    quant.append_int8(kq, ks, vq, vs, k, v, slots, bs, "bf16")
    q = _bf16(rng.standard_normal((1, 4, d)))
    out = quant.decode_int8(q, kq, ks, vq, vs, np.array([[2, 3, 4, 5, 6]]), [20], bs, "bf16")
    kd = quant.dequantize(*quant.quantize_rows(k, "bf16"))
    vd = quant.dequantize(*quant.quantize_rows(v, "bf16"))
    qf = numerics.widen(q, "bf16")
    for h in range(4):
        ref = attention.softmax_attention(qf[0, h][None], kd[:, h // 2], vd[:, h // 2],
                                          1 / np.sqrt(d))[0]
        assert np.max(np.abs(out[0, h] - ref)) < 1e-13
    # and it stays close to attention on the unquantised values (quantisation error only)
    exact = attention.softmax_attention(qf[0, 0][None], numerics.widen(k, "bf16")[:, 0],
                                        numerics.widen(v, "bf16")[:, 0], 1 / np.sqrt(d))[0]
    assert np.max(np.abs(out[0, 0] - exact)) < 0.05
