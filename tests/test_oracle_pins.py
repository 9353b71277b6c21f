"""Pins for the oracle: checks against facts the format, the pages and the
mathematics fix, chosen so that a dropped term, a wrong sign or index, or a
transposed operand in the oracle fails one of them.  CPU only."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from fp8_quantized_kv_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits(x):
    return synth.bf16_bits(torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


# ------------------------------------------------------------ e4m3 table --

def _golden_codes():
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_codes.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                parts = line.split()
                rows.append((int(parts[0], 16), float(parts[1])))
    return rows


def test_decode_matches_hand_worked_codes():
    rows = _golden_codes()
    got = oracle.e4m3_decode(np.array([c for c, _ in rows], dtype=np.uint8))
    for (code, want), g in zip(rows, got):
        if math.isnan(want):
            assert math.isnan(g), hex(code)
        else:
            assert g == want and math.copysign(1, g) == math.copysign(1, want), hex(code)


def test_decode_table_structure():
    vals = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    pos = vals[:0x7F]
    # 0x00..0x7E strictly increasing, 0x7F and 0xFF the only NaNs
    assert np.all(np.diff(pos) > 0)
    assert np.isnan(vals).sum() == 2 and np.isnan(vals[0x7F]) and np.isnan(vals[0xFF])
    # sign symmetry
    assert np.array_equal(vals[0x80:0xFF], -pos)
    # largest finite magnitude is 448 (the constant of the scale rule)
    assert np.nanmax(np.abs(vals)) == 448.0
    # subnormals: 8 values spaced 2^-9 from 0; each binade [2^e, 2^(e+1))
    # for e = -6..7 holds 8 values spaced 2^(e-3); the top binade stops at 448
    assert np.array_equal(pos[:8], np.arange(8) * 2.0 ** -9)
    for e in range(-6, 8):
        b = pos[(pos >= 2.0 ** e) & (pos < 2.0 ** (e + 1))]
        assert np.array_equal(b, 2.0 ** e + np.arange(8) * 2.0 ** (e - 3)), e
    top = pos[pos >= 256]
    assert np.array_equal(top, 256 + np.arange(7) * 32.0)
    # every value is exact in bf16 (so on-chip e4m3 -> bf16 is lossless)
    f = torch.tensor(vals[~np.isnan(vals)], dtype=torch.float64)
    assert torch.equal(f.to(torch.bfloat16).to(torch.float64), f)


def _brute_force_encode(x):
    """Nearest E4M3 value by exhaustive search; ties to the even code;
    magnitudes above 448 saturate; zero results keep the sign."""
    table = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))  # 0x00..0x7E
    a = np.abs(x.astype(np.float64))
    out = np.empty(x.shape, dtype=np.uint8)
    for i, ai in enumerate(a):
        if ai >= 448.0:
            c = 0x7E
        else:
            d = np.abs(table - ai)
            best = np.flatnonzero(d == d.min())
            c = int(best[0]) if len(best) == 1 else int(best[best % 2 == 0][0])
        out[i] = c | (0x80 if np.signbit(x[i]) else 0)
    return out


def test_encode_equals_brute_force_nearest():
    rng = np.random.default_rng(1234)
    n = 60000
    mag = 2.0 ** rng.uniform(-13, 10, n)
    x = (mag * rng.choice([-1.0, 1.0], n)).astype(np.float32)
    x = np.concatenate([x, np.float32([0.0, -0.0, 448.0, -448.0, 464.0, 1e6, -1e-30,
                                       2.0 ** -10, 2.0 ** -10 * 1.0000001])])
    assert np.array_equal(oracle.e4m3_encode(x), _brute_force_encode(x))


def test_encode_midpoints_round_to_even():
    table = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = ((table[:-1] + table[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (table[:-1] + table[1:]) / 2)  # exact
    got = oracle.e4m3_encode(mids)
    lo = np.arange(0x7E)
    want = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(got, want.astype(np.uint8))
    assert np.array_equal(oracle.e4m3_encode(-mids), (want | 0x80).astype(np.uint8))


def test_encode_decode_round_trip_all_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_encode_saturates_and_keeps_sign_of_zero():
    x = np.float32([480.0, -1e9, 449.0, 463.9, -2.0 ** -11, 2.0 ** -11, -0.0])
    assert list(oracle.e4m3_encode(x)) == [0x7E, 0xFE, 0x7E, 0x7E, 0x80, 0x00, 0x80]


# -------------------------------------------------------------- quantise --

def _worked_rows():
    rows, cur = [], {}
    with open(os.path.join(GOLDEN, "quantize_worked_row.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            cur[key] = vals
            if key == "scale_bits":
                rows.append(cur)
                cur = {}
    return rows


def test_quantize_worked_rows():
    rows = _worked_rows()
    assert len(rows) == 3
    for kv in rows:
        x = np.array([int(h, 16) for h in kv["input"]], dtype=np.uint16)[None, :]
        codes, scales = oracle.quantize(x)
        assert [int(c) for c in codes[0]] == [int(h, 16) for h in kv["codes"]]
        assert scales.view(np.uint32)[0] == int(kv["scale_bits"][0], 16)


def test_quantize_amax_element_hits_448_and_round_trip_bound():
    g = torch.Generator().manual_seed(7)
    x = (torch.randn(512, 128, generator=g) * torch.exp(torch.randn(512, 1, generator=g) * 3))
    bits = synth.bf16_bits(x.to(torch.bfloat16))
    xf = oracle.bf16_to_double(bits)
    codes, scales = oracle.quantize(bits)
    amax_idx = np.abs(xf).argmax(axis=1)
    top = codes[np.arange(512), amax_idx]
    assert np.all((top == 0x7E) | (top == 0xFE))
    assert np.all(scales == (np.abs(xf).max(axis=1).astype(np.float32) / np.float32(448)))
    deq = oracle.dequantize(codes, scales)
    # |err| <= half an E4M3 ulp of x/scale, times scale (ulp = 2^(e-3), at
    # least 2^-9 in the subnormal range), plus the fp32 rounding of x/scale
    y = np.abs(xf / scales[:, None].astype(np.float64))
    e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
    half_ulp = 2.0 ** (e - 4)
    bound = (half_ulp + y * 2.0 ** -23) * scales[:, None] * (1 + 1e-12)
    assert np.all(np.abs(deq - xf) <= bound)


def test_quantize_power_of_two_scaling():
    g = torch.Generator().manual_seed(8)
    x = torch.randn(64, 64, generator=g).to(torch.bfloat16)
    c0, s0 = oracle.quantize(synth.bf16_bits(x))
    for k in (-5, 3, 9):
        ck, sk = oracle.quantize(synth.bf16_bits(x * (2.0 ** k)))
        assert np.array_equal(ck, c0)
        assert np.array_equal(sk, s0 * np.float32(2.0 ** k))


def test_quantize_zero_row_and_single_spike():
    x = np.zeros((3, 16), dtype=np.float32)
    x[1, 5] = -3.0
    x[2, :] = 1.0
    codes, scales = oracle.quantize(_bf16_bits(x))
    assert scales[0] == 0.0 and np.all(codes[0] == 0)
    assert codes[1, 5] == 0xFE and np.all(np.delete(codes[1], 5) == 0)
    assert np.all(codes[2] == 0x7E) and scales[2] == np.float32(1.0) / np.float32(448)


# ------------------------------------------------------ pre-bias residual --

def test_residual_worked_row():
    kv = {}
    with open(os.path.join(GOLDEN, "residual_worked_row.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                key, *vals = line.split()
                kv[key] = vals
    x = np.array([int(h, 16) for h in kv["input"]], dtype=np.uint16)[None, None, :]
    b = np.array([float(v) for v in kv["bias"]], dtype=np.float32)[None, :]
    codes, scales = oracle.quantize_residual(x, b)
    assert [int(c) for c in codes[0, 0]] == [int(h, 16) for h in kv["codes"]]
    assert scales.view(np.uint32)[0, 0] == int(kv["scale_bits"][0], 16)


def test_residual_reduces_to_plain_quantisation():
    g = torch.Generator().manual_seed(15)
    # exact in bf16: small-integer residuals plus a per-head integer bias
    r = torch.randint(-40, 41, (2, 50, 128), generator=g).float()
    b = torch.randint(-64, 65, (2, 128), generator=g).float()
    k_bits = synth.bf16_bits((r + b[:, None, :]).to(torch.bfloat16))
    assert np.array_equal(oracle.bf16_to_double(k_bits), (r + b[:, None, :]).numpy())
    codes, scales = oracle.quantize_residual(k_bits, b.numpy())
    rc, rs = oracle.quantize(synth.bf16_bits(r.to(torch.bfloat16)))
    assert np.array_equal(codes, rc) and np.array_equal(scales, rs)
    # a zero bias is the plain per-row rule on the keys themselves
    c0, s0 = oracle.quantize_residual(k_bits, np.zeros((2, 128), np.float32))
    pc, ps = oracle.quantize(k_bits)
    assert np.array_equal(c0, pc) and np.array_equal(s0, ps)


def test_residual_reconstruction_bound_and_bias_exactness():
    g = torch.Generator().manual_seed(16)
    b = (torch.randn(2, 128, generator=g) * 30).float()
    k = (b[:, None, :] + torch.randn(2, 64, 128, generator=g)).to(torch.bfloat16)
    bits = synth.bf16_bits(k)
    codes, scales = oracle.quantize_residual(bits, b.numpy())
    kk = oracle.bf16_to_double(bits)
    rec = oracle.residual_keys(codes, scales, b.numpy())
    r = kk - b.numpy().astype(np.float64)[:, None, :]
    # within 1/16 of the residual's row maximum (e4m3 half-ulp at the top binade
    # is 16/448 of it) plus the fp32 rounding of the subtraction
    bound = np.abs(r).max(axis=-1, keepdims=True) / 16 + np.abs(kk) * 2.0 ** -23
    assert np.all(np.abs(rec - kk) <= bound)
    # the residual keeps far more of the token-varying part than quantising k
    plain = oracle.dequantize(*oracle.quantize(bits))
    assert np.linalg.norm(rec - kk) < 0.2 * np.linalg.norm(plain - kk)


def test_constant_key_bias_cancels_in_attention():
    # the score correction q.b is the same for every key of a row, so
    # attention over dequant(r) equals attention over dequant(r) + b
    rng = np.random.default_rng(17)
    q = rng.standard_normal((2, 8, 64))
    k = rng.standard_normal((2, 2, 40, 64))
    v = rng.standard_normal((2, 2, 40, 64))
    b = rng.standard_normal((2, 64)) * 50
    lens = np.array([40, 23], np.int32)
    a = oracle.decode_attention(q, k, v, lens, 0.125)
    c = oracle.decode_attention(q, k + b[None, :, None, :], v, lens, 0.125)
    assert np.allclose(a, c, rtol=0, atol=1e-9)


# --------------------------------------- rotated pre-bias residual (rotary) --

def _tables(P, h, angle):
    """cos and sin tables [P, h] fp32 for angle(p, i) (radians)."""
    th = np.fromfunction(angle, (P, h))
    return np.cos(th).astype(np.float32), np.sin(th).astype(np.float32)


def test_rope_bias_at_zero_angle_is_the_constant_bias():
    # cos 1, sin 0: R_t b = b exactly, so the rotated residual is the
    # constant-bias residual, bit for bit
    rng = np.random.default_rng(5)
    b = (rng.standard_normal((2, 128)) * 20).astype(np.float32)
    c, s = np.ones((64, 64), np.float32), np.zeros((64, 64), np.float32)
    pos = np.arange(40, dtype=np.int32)
    assert np.array_equal(oracle.rope_bias(b, c, s, pos), np.broadcast_to(b[:, None, :], (2, 40, 128)))
    k = _bf16_bits(rng.standard_normal((2, 40, 128)) * 4 + b[:, None, :])
    c1, s1 = oracle.quantize_residual_rope(k, b, c, s, pos)
    c0, s0 = oracle.quantize_residual(k, b)
    assert np.array_equal(c1, c0) and np.array_equal(s1.view(np.uint32), s0.view(np.uint32))
    # and a zero bias gives the plain per-row quantiser at any angle
    cr, sr = _tables(64, 64, lambda p, i: 0.37 * p + i)
    cz, sz = oracle.quantize_residual_rope(k, np.zeros((2, 128), np.float32), cr, sr, pos)
    cp, sp = oracle.quantize(k)
    assert np.array_equal(cz, cp) and np.array_equal(sz.view(np.uint32), sp.view(np.uint32))


def test_rope_bias_quarter_turn_is_rotate_half():
    # cos 0, sin 1 (a quarter turn of every pair): (R b) = (-b_hi, b_lo), the
    # "rotate half" map, exactly
    rng = np.random.default_rng(6)
    b = rng.standard_normal((3, 64)).astype(np.float32)
    c, s = np.zeros((4, 32), np.float32), np.ones((4, 32), np.float32)
    rb = oracle.rope_bias(b, c, s, np.array([0, 3], np.int32))
    want = np.concatenate([-b[:, 32:], b[:, :32]], axis=1)
    assert np.array_equal(rb[:, 0], want) and np.array_equal(rb[:, 1], want)


def test_rope_bias_is_a_rotation():
    # length kept, the inverse angle undoes it, and two rotations compose to
    # the rotation by the summed angle (each within fp32 rounding); a sign
    # error in either component breaks the last one
    rng = np.random.default_rng(7)
    b = rng.standard_normal((2, 128)).astype(np.float32)
    P, h = 50, 64
    th = rng.uniform(-math.pi, math.pi, (P, h))
    c, s = np.cos(th).astype(np.float32), np.sin(th).astype(np.float32)
    pos = np.arange(P, dtype=np.int32)
    rb = oracle.rope_bias(b, c, s, pos).astype(np.float64)
    assert np.allclose(np.linalg.norm(rb, axis=-1), np.linalg.norm(b, axis=-1)[:, None], rtol=1e-6)
    for t in (0, 17, 49):
        back = oracle.rope_bias(rb[:, t].astype(np.float32), c[t:t + 1], -s[t:t + 1], np.zeros(1, np.int32))
        assert np.allclose(back[:, 0], b, atol=1e-5)
        th2 = rng.uniform(-math.pi, math.pi, h)
        c2, s2 = np.cos(th2).astype(np.float32)[None], np.sin(th2).astype(np.float32)[None]
        two = oracle.rope_bias(rb[:, t].astype(np.float32), c2, s2, np.zeros(1, np.int32))[:, 0]
        cs = np.cos(th[t] + th2).astype(np.float32)[None]
        sn = np.sin(th[t] + th2).astype(np.float32)[None]
        one = oracle.rope_bias(b, cs, sn, np.zeros(1, np.int32))[:, 0]
        assert np.allclose(two, one, atol=1e-5)


def test_rope_residual_reconstruction_bound():
    # dequant(r) + R_t b stays within the residual's quantisation error of
    # the key, and keeps the token-varying part that a plain quantiser of the
    # biased key loses
    rng = np.random.default_rng(8)
    P, h = 80, 64
    c, s = _tables(P, h, lambda p, i: p * 10000.0 ** (-i / h))
    b = np.zeros((2, 128), np.float32)
    b[:, :4] = 60.0
    pos = np.arange(P, dtype=np.int32)
    rb = oracle.rope_bias(b, c, s, pos)
    kf = rng.standard_normal((2, P, 128)).astype(np.float32) + rb
    k = _bf16_bits(kf)
    codes, scales = oracle.quantize_residual_rope(k, b, c, s, pos)
    rec = oracle.residual_rope_keys(codes, scales, rb)
    kd = oracle.bf16_to_double(k)
    resid = kd - rb
    amax = np.abs(resid).max(axis=-1, keepdims=True)
    assert np.all(np.abs(rec - kd) <= amax / 16 + 1e-12)
    plain = oracle.dequantize(*oracle.quantize(k))
    assert np.linalg.norm(rec - kd) < 0.5 * np.linalg.norm(plain - kd)


# ----------------------------------------------------------------- MXFP8 --

def _mx_worked_row():
    kv = {}
    with open(os.path.join(GOLDEN, "mx_quantize_worked_row.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                key, *vals = line.split()
                kv[key] = [int(h, 16) for h in vals]
    return kv


def test_mx_quantize_worked_row():
    kv = _mx_worked_row()
    assert len(kv["input"]) == 128 and len(kv["codes"]) == 128 and len(kv["e8m0"]) == 4
    codes, scales = oracle.mx_quantize(np.array(kv["input"], dtype=np.uint16)[None, :])
    assert [int(c) for c in codes[0]] == kv["codes"]
    assert [int(b) for b in scales[0]] == kv["e8m0"]


def _mx_rows(seed, n=256, d=128):
    """bf16 rows whose 32-element blocks span 2^-140 .. 2^120 in magnitude,
    with zero blocks, single spikes and bf16 subnormals."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, d, generator=g) * torch.exp2(torch.randint(-140, 120, (n, d // 32), generator=g)
                                                  .float().repeat_interleave(32, dim=1))
    x[::17, :32] = 0.0
    x[5::23, 40] = 1e30
    return synth.bf16_bits(x.to(torch.bfloat16))


def test_mx_scale_is_the_smallest_power_of_two_that_fits():
    bits = _mx_rows(11)
    x = oracle.bf16_to_double(bits).reshape(-1, 4, 32)
    _, scales = oracle.mx_quantize(bits)
    E = scales.reshape(-1, 4).astype(np.int64) - 127
    amax = np.abs(x).max(axis=-1)
    X = np.ldexp(1.0, E)
    assert np.all(amax <= 448.0 * X)
    nz = amax > 0
    # one power of two smaller would overflow 448 (unless E is already -127)
    assert np.all((amax[nz] > 448.0 * X[nz] / 2) | (E[nz] == -127))
    assert np.all(E[~nz] == -127)


def test_mx_elements_are_nearest_e4m3_of_the_scaled_value():
    bits = _mx_rows(12)
    x = oracle.bf16_to_double(bits)
    codes, scales = oracle.mx_quantize(bits)
    X = np.ldexp(1.0, scales.astype(np.int64) - 127).repeat(32, axis=-1)
    deq = oracle.mx_dequantize(codes, scales)
    assert np.array_equal(deq, oracle.e4m3_decode(codes) * X)
    # brute force: the dequantised value is a nearest E4M3 grid point of x/X
    grid = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    grid = np.unique(grid[np.isfinite(grid)])
    y = (x / X).ravel()
    d_best = np.abs(grid[None, :] - y[:, None]).min(axis=1)
    got = (deq / X).ravel()
    # fp32 rounding of x * 2^-E only matters below the fp32 normal range
    assert np.all(np.abs(got - y) <= d_best * (1 + 1e-12) + 2.0 ** -149)
    # and never beyond half the top binade's spacing (16) times X
    assert np.all(np.abs(deq - x) <= 16 * X)


def test_mx_round_trip_is_exact_on_the_grid():
    bits = _mx_rows(13)
    codes, scales = oracle.mx_quantize(bits)
    deq = oracle.mx_dequantize(codes, scales)
    again = synth.bf16_bits(torch.from_numpy(deq).to(torch.bfloat16))
    assert np.array_equal(oracle.bf16_to_double(again), deq)        # the grid fits in bf16 here
    c2, s2 = oracle.mx_quantize(again)
    assert np.array_equal(oracle.mx_dequantize(c2, s2), deq)


def test_mx_scaling_by_powers_of_two_moves_only_the_scale():
    g = torch.Generator().manual_seed(14)
    x = torch.randn(32, 128, generator=g).to(torch.bfloat16)
    c0, s0 = oracle.mx_quantize(synth.bf16_bits(x))
    for k in (-20, -3, 5, 40):
        ck, sk = oracle.mx_quantize(synth.bf16_bits(x * (2.0 ** k)))
        assert np.array_equal(ck, c0)
        assert np.array_equal(sk.astype(int), s0.astype(int) + k)


# ------------------------------------------------------------- attention --

def _brute_attention(q, k, v, sm_scale):
    """Full score matrix and a softmax without max shift in extended precision."""
    ql = q.astype(np.longdouble)
    kl = k.astype(np.longdouble)
    vl = v.astype(np.longdouble)
    s = (ql @ kl.T) * np.longdouble(sm_scale)
    w = np.exp(s)
    w = w / w.sum(axis=-1, keepdims=True)
    return (w @ vl).astype(np.float64)


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_decode_equals_brute_force():
    B, Hq, Hkv, T, D = 2, 6, 2, 9, 8
    q, k, v = _rand((B, Hq, D), 1), _rand((B, Hkv, T, D), 2), _rand((B, Hkv, T, D), 3)
    lens = np.array([9, 4], dtype=np.int32)
    out = oracle.decode_attention(q, k, v, lens, 0.37)
    for b in range(B):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            ref = _brute_attention(q[b, h][None], k[b, g, :lens[b]], v[b, g, :lens[b]], 0.37)[0]
            assert np.max(np.abs(out[b, h] - ref)) < 1e-12


def test_softmax_weights_sum_to_one():
    T = D = 12
    q = _rand((1, 1, D), 4) * 3
    k = _rand((1, 1, T, D), 5)
    v = np.eye(T)[None, None]          # one-hot values: o is the weight vector
    o = oracle.decode_attention(q, k, v, np.array([T], np.int32), 0.5)[0, 0]
    assert abs(o.sum() - 1.0) < 1e-12 and np.all(o > 0)
    w = _brute_attention(q[0], k[0, 0], np.eye(T), 0.5)[0]
    assert np.max(np.abs(o - w)) < 1e-12


def test_closed_forms():
    D = 16
    q = _rand((1, 2, D), 6)
    v = _rand((1, 1, 5, D), 7)
    # one key: output is that key's value
    o = oracle.decode_attention(q, _rand((1, 1, 5, D), 8), v, np.array([1], np.int32), 1.0)
    assert np.array_equal(o[0, 0], v[0, 0, 0]) and np.array_equal(o[0, 1], v[0, 0, 0])
    # all keys equal: output is the mean value
    k = np.repeat(_rand((1, 1, 1, D), 9), 5, axis=2)
    o = oracle.decode_attention(q, k, v, np.array([5], np.int32), 1.0)
    assert np.max(np.abs(o[0, 0] - v[0, 0].mean(axis=0))) < 1e-12
    # zero length: zero output
    o = oracle.decode_attention(q, k, v, np.array([0], np.int32), 1.0)
    assert np.all(o == 0)


def test_key_shift_invariance():
    D, T = 32, 40
    q = _rand((1, 3, D), 10)
    k = _rand((1, 1, T, D), 11)
    v = _rand((1, 1, T, D), 12)
    c = _rand((D,), 13) * 5
    lens = np.array([T], np.int32)
    o1 = oracle.decode_attention(q, k, v, lens, 0.2)
    o2 = oracle.decode_attention(q, k + c, v, lens, 0.2)
    assert np.max(np.abs(o1 - o2)) < 1e-12


def test_gqa_equals_mha_with_repeated_heads():
    B, Hq, Hkv, T, D = 2, 8, 2, 30, 16
    q = _rand((B, Hq, D), 14)
    k = _rand((B, Hkv, T, D), 15)
    v = _rand((B, Hkv, T, D), 16)
    lens = np.array([30, 17], np.int32)
    gqa = oracle.decode_attention(q, k, v, lens, 0.25)
    G = Hq // Hkv
    mha = oracle.decode_attention(q, np.repeat(k, G, axis=1), np.repeat(v, G, axis=1), lens, 0.25)
    assert np.array_equal(gqa, mha)
    # and head h really reads KV head h // G (not h % Hkv)
    wrong = oracle.decode_attention(q, np.tile(k, (1, G, 1, 1)), np.tile(v, (1, G, 1, 1)), lens, 0.25)
    assert not np.allclose(gqa, wrong)


def test_prefill_rows_equal_decode_prefixes_and_brute_force():
    n_q, pos0, Hq, Hkv, D = 7, 5, 4, 2, 8
    Tk = pos0 + n_q
    q = _rand((n_q, Hq, D), 17)
    k = _rand((Hkv, Tk, D), 18)
    v = _rand((Hkv, Tk, D), 19)
    out = oracle.prefill_attention(q, k, v, pos0, 0.3)
    for i in range(n_q):
        n = pos0 + i + 1
        dec = oracle.decode_attention(q[i][None], k[None], v[None], np.array([n], np.int32), 0.3)[0]
        assert np.array_equal(out[i], dec)
        for h in range(Hq):
            g = h // (Hq // Hkv)
            ref = _brute_attention(q[i, h][None], k[g, :n], v[g, :n], 0.3)[0]
            assert np.max(np.abs(out[i, h] - ref)) < 1e-12
    # causality: changing a key after position pos0+i leaves row i unchanged
    k2 = k.copy()
    k2[:, pos0 + 3:] += 10
    out2 = oracle.prefill_attention(q, k2, v, pos0, 0.3)
    assert np.array_equal(out[:3], out2[:3]) and not np.allclose(out[3:], out2[3:])


# ----------------------------------------------------------------- paged --

def test_gather_paged():
    P, heads, num_pages, D = 4, 2, 6, 3
    pool = np.arange(num_pages * heads * P * D, dtype=np.float32).reshape(num_pages, heads, P, D)
    table = np.array([[5, 0, 3], [1, 2, -1]], dtype=np.int32)
    out = oracle.gather_paged(pool, table, 0, 10)
    assert out.shape == (heads, 10, D)
    # token 6 of sequence 0: page table[0][1] = 0, offset 2
    assert np.array_equal(out[1, 6], pool[0, 1, 2])
    assert np.array_equal(out[0, 9], pool[3, 0, 1])
    ident = np.arange(num_pages, dtype=np.int32)[None]
    assert np.array_equal(oracle.gather_paged(pool, ident, 0, num_pages * P),
                          pool.transpose(1, 0, 2, 3).reshape(heads, num_pages * P, D))
    with pytest.raises(ValueError):
        oracle.gather_paged(pool, table, 1, 9)     # reaches the -1 entry


# ------------------------------------------------- the gate has teeth --

def test_gate_rejects_broken_scales():
    """"FP8 KV cache (fp8_kv, opt-in)", bullet "Accuracy": a V scale x1.05 and
    one token's scale used for every token must both fail the gate."""
    spec = synth.WORKLOADS["decode_b16_ctx512"]
    inp = synth.decode_inputs(spec, seq_lens=[512] * 2)
    B, Hkv, D = 2, spec.kv_heads, spec.head_dim
    T = 512
    kb = synth.bf16_bits(inp.k).reshape(B, T, Hkv, D).transpose(0, 2, 1, 3)
    vb = synth.bf16_bits(inp.v).reshape(B, T, Hkv, D).transpose(0, 2, 1, 3)
    q = oracle.bf16_to_double(synth.bf16_bits(inp.q[:B]))
    kc, ks = oracle.quantize(kb)
    vc, vs = oracle.quantize(vb)
    lens = np.full(B, T, np.int32)
    sm = 1 / math.sqrt(D)
    ref = oracle.decode_attention(q, oracle.dequantize(kc, ks), oracle.dequantize(vc, vs), lens, sm)
    same = oracle.decode_attention(q, oracle.dequantize(kc, ks), oracle.dequantize(vc, vs), lens, sm)
    assert oracle.attention_gate(same, ref)[0]
    bad_v = oracle.decode_attention(q, oracle.dequantize(kc, ks), oracle.dequantize(vc, vs * 1.05), lens, sm)
    assert not oracle.attention_gate(bad_v, ref)[0]
    one = np.broadcast_to(ks[..., :1], ks.shape)
    bad_k = oracle.decode_attention(q, oracle.dequantize(kc, one), oracle.dequantize(vc, vs), lens, sm)
    assert not oracle.attention_gate(bad_k, ref)[0]


def test_fp8_kv_error_zero_on_exact_cache_and_small_otherwise():
    # rows whose values are E4M3 numbers with amax 448: quantisation is exact
    rng = np.random.default_rng(3)
    table = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    k = rng.choice(table[table <= 448], size=(1, 1, 20, 16)) * rng.choice([-1, 1], size=(1, 1, 20, 16))
    v = rng.choice(table[table <= 448], size=(1, 1, 20, 16))
    k[..., 0] = 448.0
    v[..., 0] = -448.0
    q = rng.standard_normal((1, 2, 16)) * 0.01
    err = oracle.fp8_kv_error(_bf16_bits(q), _bf16_bits(k), _bf16_bits(v), np.array([20], np.int32), 0.25)
    assert err == 0.0
    g = torch.Generator().manual_seed(0)
    q = torch.randn(2, 4, 64, generator=g).to(torch.bfloat16)
    k = torch.randn(2, 1, 128, 64, generator=g).to(torch.bfloat16)
    v = torch.randn(2, 1, 128, 64, generator=g).to(torch.bfloat16)
    err = oracle.fp8_kv_error(synth.bf16_bits(q), synth.bf16_bits(k), synth.bf16_bits(v),
                              np.array([77, 128], np.int32), 0.125)
    assert 1e-3 < err < 5e-2
