"""Pins for the oracle's numeric building blocks, against library routines,
closed forms, invariants and brute force (never against a retyped formula)."""
import math

import numpy as np
import pytest

from oracle import model as M

torch = pytest.importorskip("torch")
rng = np.random.default_rng(1234)


def test_bf16_matches_torch_cast_on_float32_values():
    x = rng.standard_normal(5000).astype(np.float32) * np.float32(5.0)
    # exact ties between neighbouring bfloat16 values, both parities
    ties = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 3 * 2 ** -9 * (1 + 2 ** -8)])
    x = np.concatenate([x.astype(np.float64), ties])
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(M.bf16(x), ref)
    assert M.bf16(1 + 2 ** -8) == 1.0                   # tie -> even (1.0)
    assert M.bf16(1 + 3 * 2 ** -8) == 1 + 2 ** -6       # tie -> even (1 + 2^-6)
    assert M.bf16(0.0) == 0.0


def test_bf16_direct_from_float64_no_double_rounding():
    # 1 + 2^-8 + 2^-30 is just above the tie: nearest bf16 is 1 + 2^-7.
    # Through float32 it would first round to the tie 1 + 2^-8, then to even 1.0.
    x = 1 + 2 ** -8 + 2 ** -30
    assert M.bf16(x) == 1 + 2 ** -7


def test_rms_norm_matches_torch():
    x = rng.standard_normal((7, 96))
    g = rng.standard_normal(96)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (96,), torch.from_numpy(g), eps=1e-5)
    np.testing.assert_allclose(M.rms_norm(x, g, 1e-5), ref.numpy(), rtol=1e-13, atol=1e-14)


def test_linear_matches_brute_force():
    x = rng.standard_normal((3, 5))
    w = rng.standard_normal((4, 5)).astype(np.float32)
    b = rng.standard_normal(4)
    ref = np.array([[sum(float(x[i, k]) * float(w[o, k]) for k in range(5)) + b[o] for o in range(4)]
                    for i in range(3)])
    np.testing.assert_allclose(M.linear(x, w, b, block=3), ref, rtol=1e-14)


def test_rope_closed_form_small():
    # d_h = 4: pair (0, 2) rotates at theta^0 = 1 rad per position, pair (1, 3) at theta^(-1/2).
    theta = 100.0
    x = np.array([[[1.0, 2.0, 3.0, 4.0]]])
    out = M.rope(x, np.array([3]), theta)[0, 0]
    a0, a1 = 3.0, 3.0 / 10.0
    exp = [1 * math.cos(a0) - 3 * math.sin(a0), 2 * math.cos(a1) - 4 * math.sin(a1),
           3 * math.cos(a0) + 1 * math.sin(a0), 4 * math.cos(a1) + 2 * math.sin(a1)]
    np.testing.assert_allclose(out, exp, rtol=1e-14)


def test_rope_complex_form_and_invariants():
    n, h, d_h, theta = 9, 3, 16, 10000.0
    x = rng.standard_normal((n, h, d_h))
    pos = rng.integers(0, 5000, n)
    out = M.rope(x, pos, theta)
    # same rotation written as complex multiplication of (x_i + i x_{i+d/2})
    z = x[..., : d_h // 2] + 1j * x[..., d_h // 2:]
    freq = theta ** (-np.arange(d_h // 2) * 2.0 / d_h)
    zr = z * np.exp(1j * pos[:, None, None] * freq[None, None, :])
    np.testing.assert_allclose(out, np.concatenate([zr.real, zr.imag], axis=-1), rtol=1e-9, atol=1e-12)
    # position 0 is the identity; rotation preserves norms
    np.testing.assert_array_equal(M.rope(x, np.zeros(n, int), theta), x)
    np.testing.assert_allclose(np.linalg.norm(out, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-12)
    # relative-position property: <R(p) q, R(p') k> depends only on p - p'
    q = rng.standard_normal((1, 1, d_h))
    k = rng.standard_normal((1, 1, d_h))
    dots = [float((M.rope(q, np.array([p + 7]), theta) * M.rope(k, np.array([p]), theta)).sum())
            for p in (0, 13, 400, 3001)]
    np.testing.assert_allclose(dots, dots[0], rtol=1e-9)


def test_attention_matches_torch_sdpa_gqa():
    n, n_q, n_kv, d_h = 37, 8, 2, 16
    q = rng.standard_normal((n, n_q, d_h))
    k = rng.standard_normal((n, n_kv, d_h))
    v = rng.standard_normal((n, n_kv, d_h))
    pos = np.arange(n)
    got = M.causal_gqa_attention(q, k, v, pos, pos)
    tq, tk, tv = (torch.from_numpy(a).permute(1, 0, 2)[None] for a in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True, enable_gqa=True)
    np.testing.assert_allclose(got, ref[0].permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)


def test_attention_brute_force_decode_rows():
    # one query at position 5 over keys 0..7 (keys 6, 7 must be masked)
    n_q, n_kv, d_h = 4, 2, 3
    q = rng.standard_normal((1, n_q, d_h))
    k = rng.standard_normal((8, n_kv, d_h))
    v = rng.standard_normal((8, n_kv, d_h))
    got = M.causal_gqa_attention(q, k, v, np.array([5]), np.arange(8))
    for h in range(n_q):
        kv = h // 2
        s = [sum(q[0, h, c] * k[t, kv, c] for c in range(d_h)) / math.sqrt(d_h) for t in range(6)]
        e = [math.exp(a - max(s)) for a in s]
        ref = [sum(e[t] * v[t, kv, c] for t in range(6)) / sum(e) for c in range(d_h)]
        np.testing.assert_allclose(got[0, h], ref, rtol=1e-12)


def test_attention_zero_query_is_causal_running_mean():
    n, d_h = 6, 4
    v = rng.standard_normal((n, 1, d_h))
    out = M.causal_gqa_attention(np.zeros((n, 2, d_h)), rng.standard_normal((n, 1, d_h)), v,
                                 np.arange(n), np.arange(n))
    run_mean = np.cumsum(v[:, 0], axis=0) / np.arange(1, n + 1)[:, None]
    np.testing.assert_allclose(out[:, 0], run_mean, rtol=1e-13)
    np.testing.assert_allclose(out[:, 1], run_mean, rtol=1e-13)


def test_silu_special_values():
    assert M.silu(np.float64(0.0)) == 0.0
    np.testing.assert_allclose(M.silu(np.float64(40.0)), 40.0, rtol=1e-15)
    np.testing.assert_allclose(M.silu(np.float64(1.0)), 1.0 / (1.0 + math.exp(-1.0)), rtol=1e-15)
    x = torch.linspace(-8, 8, 101, dtype=torch.float64)
    np.testing.assert_allclose(M.silu(x.numpy()), torch.nn.functional.silu(x).numpy(), rtol=1e-14)


def test_compute_in_float32_linear():
    """The precision switch used to measure the float32 floor: inside it the linear layer is a
    float32 matmul of the same (bfloat16-valued) operands, its bias added in float32."""
    x = M.bf16(rng.standard_normal((5, 64)))
    w = M.bf16(rng.standard_normal((7, 64))).astype(np.float32)
    b = rng.standard_normal(7) * 0.1
    exact = M.linear(x, w, b)
    with M.compute_in(np.float32):
        f32 = M.linear(x, w, b)
    want = ((x.astype(np.float32) @ w.T) + b.astype(np.float32)).astype(np.float64)
    assert np.array_equal(f32, want)
    assert not np.array_equal(f32, exact)
    np.testing.assert_allclose(f32, exact, rtol=1e-5, atol=1e-5)
    assert np.array_equal(M.linear(x, w, b), exact)      # switch restored


def test_compute_in_float32_attention():
    """Inside the switch the attention is a float32 evaluation: scores, scaling, max, exp,
    normaliser and weighted sum of V, each in float32 (brute-force loops on a tiny case);
    outside it the float64 definition is untouched."""
    n_q, d_h = 2, 4
    q = M.bf16(rng.standard_normal((3, n_q, d_h)))
    k = M.bf16(rng.standard_normal((3, 1, d_h)))
    v = M.bf16(rng.standard_normal((3, 1, d_h)))
    pos = np.arange(3)
    exact = M.causal_gqa_attention(q, k, v, pos, pos)
    with M.compute_in(np.float32):
        got = M.causal_gqa_attention(q, k, v, pos, pos)
    f32 = np.float32
    sc = f32(1.0 / math.sqrt(d_h))
    for h in range(n_q):
        for i in range(3):
            s = []
            for t in range(i + 1):
                acc = f32(0)
                for e in range(d_h):
                    acc = f32(acc + f32(q[i, h, e]) * f32(k[t, 0, e]))
                s.append(f32(acc * sc))
            mx = max(s)
            w = [np.exp(f32(a - mx)) for a in s]
            den = f32(0)
            for t in range(i + 1):
                den = f32(den + w[t])
            for e in range(d_h):
                num = f32(0)
                for t in range(i + 1):
                    num = f32(num + w[t] * f32(v[t, 0, e]))
                np.testing.assert_allclose(got[i, h, e], float(f32(num / den)), rtol=2e-6, atol=1e-7)
    assert not np.array_equal(got, exact)
    np.testing.assert_allclose(got, exact, rtol=1e-5, atol=1e-6)
    assert np.array_equal(M.causal_gqa_attention(q, k, v, pos, pos), exact)   # switch restored


def test_compute_in_float32_pointwise_ops():
    """RMSNorm (mean of squares, reciprocal root, scaling), RoPE (float64 angles, float32
    rotation), SiLU, the SwiGLU product and the residual add, each against a direct float32
    evaluation, and untouched outside the switch."""
    f32 = np.float32
    x = rng.standard_normal((4, 64)) * 0.3
    g = 1.0 + 0.1 * rng.standard_normal(64)
    ref = M.rms_norm(x, g, 1e-5)
    with M.compute_in(np.float32):
        r32 = M.rms_norm(x, g, 1e-5)
        xs = rng.standard_normal((3, 2, 8))
        ro = M.rope(xs, np.array([0, 5, 1000]), 10000.0)
        sl = M.silu(x)
        sw = M.swiglu(x, x[::-1])
        ra = M.residual_add(x, x * 1e-3)
    xt = x.astype(f32)
    ms = np.mean(xt * xt, axis=-1, keepdims=True, dtype=f32)
    np.testing.assert_array_equal(r32, (xt * (f32(1) / np.sqrt(ms + f32(1e-5))) * g.astype(f32)).astype(np.float64))
    np.testing.assert_allclose(r32, ref, rtol=1e-6)
    assert np.array_equal(M.rms_norm(x, g, 1e-5), ref)
    inv = np.power(10000.0, -2.0 * np.arange(4) / 8)
    ang = np.array([0, 5, 1000])[:, None] * inv[None, :]
    c, s_ = np.cos(ang).astype(f32)[:, None, :], np.sin(ang).astype(f32)[:, None, :]
    a1, a2 = xs[..., :4].astype(f32), xs[..., 4:].astype(f32)
    np.testing.assert_array_equal(ro, np.concatenate([a1 * c - a2 * s_, a2 * c + a1 * s_], axis=-1).astype(np.float64))
    np.testing.assert_array_equal(sl, (xt / (f32(1) + np.exp(-xt))).astype(np.float64))
    np.testing.assert_array_equal(sw, ((xt / (f32(1) + np.exp(-xt))) * x[::-1].astype(f32)).astype(np.float64))
    np.testing.assert_array_equal(ra, (xt + (x * 1e-3).astype(f32)).astype(np.float64))
    assert np.array_equal(M.silu(x), x / (1.0 + np.exp(-x)))


def test_e4m3_matches_torch_float8_cast():
    """float8 e4m3 rounding against torch's float8_e4m3fn cast (round to nearest even)
    over normals, subnormals, exact ties and values just below powers of two."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.uniform(-448, 448, 4000), rng.uniform(-1, 1, 4000) * 2.0 ** rng.integers(-12, 0, 4000),
        np.array([0.0, 1.0625, 1.1875, -1.1875, 2 ** -10, 3 * 2 ** -10, 5 * 2 ** -11, 2 ** -6, 255.99, 447.9,
                  np.nextafter(256.0, 0.0), np.nextafter(2.0 ** -6, 0.0)])]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(M.e4m3(x.astype(np.float64)), ref)


def test_e4m3_grid_by_hand():
    # 4 significant bits: 1, 1.125, ..., 1.875 between 1 and 2; 2^-9 steps below 2^-6
    assert M.e4m3(1.0625) == 1.0 and M.e4m3(1.1875) == 1.25 and M.e4m3(1.2) == 1.25
    assert M.e4m3(17.0) == 16.0 and M.e4m3(17.5) == 18.0
    assert M.e4m3(2 ** -10) == 0.0 and M.e4m3(3 * 2 ** -10) == 2 ** -8
    assert M.e4m3(500.0) == 448.0 and M.e4m3(-1e9) == -448.0


def test_fp8_quantize_per_token_and_head():
    """One scale per (token, head) vector: the largest magnitude maps to +-448 exactly,
    every code is an e4m3 value, dequantized values are within half an e4m3 step, a zero
    vector stays zero, and quantization is per vector (scaling one vector changes only its
    own scale)."""
    rng = np.random.default_rng(9)
    v = M.bf16(rng.normal(0, 1, (5, 3, 64)) * np.array([1e-3, 1.0, 50.0])[None, :, None])
    v[2, 1] = 0.0
    codes, scale = M.fp8_quantize(v)
    assert scale.shape == (5, 3) and scale.dtype == np.float32
    np.testing.assert_array_equal(M.e4m3(codes), codes)
    amax = np.abs(codes).max(axis=-1)
    assert np.all(amax[scale > 0] == 448.0) and scale[2, 1] == 0 and np.all(codes[2, 1] == 0)
    deq = M.fp8_dequantize(codes, scale)
    step = np.exp2(np.floor(np.log2(np.maximum(np.abs(codes), 2 ** -6))) - 3) * scale[..., None]
    assert np.all(np.abs(deq - v) <= 0.5 * step * (1 + 1e-6) + 1e-12)
    v2 = v.copy()
    v2[0, 0] *= 4.0
    c2, s2 = M.fp8_quantize(v2)
    assert s2[0, 0] == np.float32(scale[0, 0] * 4) and np.array_equal(s2[1:], scale[1:])
    np.testing.assert_array_equal(c2[1:], codes[1:])
