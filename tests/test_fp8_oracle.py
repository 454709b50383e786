"""Pins of the FP8 oracle (CPU): the e4m3 format against torch's float8_e4m3fn
conversion and the format's definition, the Hadamard rotation against
scipy's Sylvester matrix and its invariance, quantisation round trips, the
forward's exact cases and its error bound; then planted mistakes, each of
which must fail one pin."""
import copy
import math
import types

import numpy as np
import pytest
import scipy.linalg
import torch

import oracle.fp8_ref as fp8

# ---------------------------------------------------------------------------
# Pins (each takes the module under test)
# ---------------------------------------------------------------------------


def _all_e4m3_values():
    v = np.array([np.ldexp(1.0 + m / 8.0, e - 7) for e in range(1, 16) for m in range(8) if not (e == 15 and m == 7)]
                 + [np.ldexp(m / 8.0, -6) for m in range(8)])
    return np.sort(np.concatenate([v, -v]))


def pin_round_matches_torch(ref):
    """RNE rounding of float32 values below the saturation range equals torch's
    float8_e4m3fn conversion (random values over all binades, every e4m3 value,
    and every midpoint between neighbours, i.e. all ties)."""
    rng = np.random.default_rng(3)
    vals = _all_e4m3_values()
    pos = np.unique(vals[vals >= 0])
    mids = (pos[:-1] + pos[1:]) / 2
    rnd = np.ldexp(rng.uniform(1, 2, 20000), rng.integers(-12, 9, 20000)) * rng.choice([-1, 1], 20000)
    x = np.concatenate([vals, mids, -mids, rnd]).astype(np.float32)
    x = x[np.abs(x) < 464]
    got = ref.e4m3_round(x.astype(np.float64))
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(got, want)


def pin_saturation_and_codes(ref):
    """Values past 448 saturate (the PTX satfinite rule); decode(encode(v)) = v
    for every finite code, and the named codes have the format's values."""
    assert np.array_equal(ref.e4m3_round(np.array([464.0, 1e6, -500.0])), [448.0, 448.0, -448.0])
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    vals = ref.e4m3_decode(codes)
    assert np.array_equal(ref.e4m3_decode(ref.e4m3_encode(vals)), vals)
    assert np.array_equal(ref.e4m3_encode(vals)[vals != 0], codes[vals != 0])
    named = {0x7E: 448.0, 0x08: 2.0 ** -6, 0x01: 2.0 ** -9, 0x38: 1.0, 0xB8: -1.0, 0x07: 7 * 2.0 ** -9}
    for c, v in named.items():
        assert ref.e4m3_decode(np.array([c], dtype=np.uint8))[0] == v, hex(c)
    assert np.isnan(ref.e4m3_decode(np.array([0x7F], dtype=np.uint8))[0])


def pin_fwht_is_sylvester(ref):
    """fwht_f32(x) = x H_d with H_d the Sylvester-Hadamard matrix (scipy), and
    the rotation is orthogonal: it keeps q.k (fp64 products of the fp32 outputs)."""
    rng = np.random.default_rng(4)
    for d in (8, 16, 64, 128, 256):
        x = rng.standard_normal((5, d)).astype(np.float32)
        want = x.astype(np.float64) @ scipy.linalg.hadamard(d)
        assert np.max(np.abs(ref.fwht_f32(x) - want)) <= 1e-5 * np.abs(want).max()
        eye = np.eye(d, dtype=np.float32)
        assert np.array_equal(ref.fwht_f32(eye), scipy.linalg.hadamard(d).astype(np.float32))
        q = rng.standard_normal((7, d)).astype(np.float32)
        k = rng.standard_normal((9, d)).astype(np.float32)
        qr = ref.incoherent_rotate_f32(q, 12345).astype(np.float64)
        kr = ref.incoherent_rotate_f32(k, 12345).astype(np.float64)
        qk = q.astype(np.float64) @ k.astype(np.float64).T
        assert np.max(np.abs(qr @ kr.T - qk)) <= 1e-5 * (1 + np.abs(qk).max())
        s = ref.hadamard_signs(d, 12345)
        assert set(np.unique(s)) <= {-1.0, 1.0} and 0 < (s < 0).sum() < d
    # past 128 columns the signs continue from the next counter block: the
    # first 128 of d = 256 are those of d = 128, the rest a different draw
    s256, s128 = ref.hadamard_signs(256, 777), ref.hadamard_signs(128, 777)
    assert np.array_equal(s256[:128], s128) and not np.array_equal(s256[128:], s128)


def pin_quantize_round_trip(ref):
    """Per-head quantisation: amax maps to 448 exactly, every element comes back
    within half an e4m3 unit (2^-4 relative, 2^-10 descale among subnormals),
    an all-zero head gets descale 1, and the transposed layout is the transpose."""
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((2, 3, 50, 64)) * rng.uniform(0.1, 10, (2, 3, 1, 1))).astype(np.float32)
    x[1, 2] = 0
    codes, ds = ref.fp8_quantize_ref(x)
    back = ref.fp8_dequantize(codes, ds)
    err = np.abs(back - x)
    lim = np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10 * ds[:, :, None, None]) * (1 + 1e-6)
    assert np.all(err <= lim)
    assert ds[1, 2] == 1.0 and np.all(codes[1, 2] == 0)
    for b in range(2):
        for h in range(3):
            if (b, h) != (1, 2):
                assert np.max(np.abs(ref.e4m3_decode(codes[b, h]))) == 448.0
    ct, dst = ref.fp8_quantize_ref(x, transpose=True)
    assert np.array_equal(ct, np.swapaxes(codes, -1, -2)) and np.array_equal(dst, ds)


def _fp8_case(ref, B, H, N, d, seed, causal, qk=1.0):
    rng = np.random.default_rng(seed)
    q, k, v = (rng.standard_normal((B, H, N, d)).astype(np.float32) for _ in range(3))
    q8, dq = ref.fp8_quantize_ref(q * qk)
    k8, dk = ref.fp8_quantize_ref(k * qk)
    vt8, dv = ref.fp8_quantize_ref(v, transpose=True)
    return ref.attn_fwd_fp8_ref(q8, k8, vt8, dq, dk, dv, 1 / math.sqrt(d), causal), (q8, k8, vt8, dq, dk, dv)


def pin_fp8_forward_exact_parts(ref):
    """O_exact and LSE are the plain definition on the dequantised inputs
    (scipy softmax and logsumexp); the rounded forward stays inside its bound
    and the bound is not vacuous (well under the output scale)."""
    from scipy.special import logsumexp, softmax
    for causal in (False, True):
        (O, LSE, O8, bound), (q8, k8, vt8, dq, dk, dv) = _fp8_case(ref, 1, 2, 40, 16, 6 + causal, causal, qk=2.0)
        Q, K = ref.fp8_dequantize(q8, dq), ref.fp8_dequantize(k8, dk)
        V = np.swapaxes(ref.fp8_dequantize(vt8, dv), -1, -2)
        for h in range(2):
            S = (Q[0, h] @ K[0, h].T) / 4.0
            if causal:
                S = np.where(np.tril(np.ones_like(S)) > 0, S, -np.inf)
            assert np.max(np.abs(O[0, h] - softmax(S, axis=1) @ V[0, h])) <= 1e-12
            assert np.max(np.abs(LSE[0, h] - logsumexp(S, axis=1))) <= 1e-12
        assert np.all(np.abs(O8 - O) <= bound * (1 + 1e-9))
        assert np.max(bound) <= 0.1 * np.max(np.abs(V)) and np.max(np.abs(O8 - O)) > 0


def pin_fp8_power_of_two_probabilities(ref):
    """Scores whose exponentials are powers of two (scale ln 2, integer q.k) give
    probabilities e4m3 holds exactly: the rounded forward equals the exact one."""
    B, H, N, d = 1, 1, 12, 16
    rng = np.random.default_rng(7)
    q8 = np.zeros((B, H, N, d), dtype=np.uint8)
    q8[..., 0] = ref.e4m3_encode(np.array([1.0]))[0]
    a = rng.integers(0, 9, N).astype(np.float64)
    k8 = np.zeros((B, H, N, d), dtype=np.uint8)
    k8[0, 0, :, 0] = ref.e4m3_encode(-a)
    vt8, dv = ref.fp8_quantize_ref(rng.standard_normal((B, H, N, d)).astype(np.float32), transpose=True)
    one = np.ones((B, H), dtype=np.float32)
    O, LSE, O8, _ = ref.attn_fwd_fp8_ref(q8, k8, vt8, one, one, dv, math.log(2.0), False)
    assert np.max(np.abs(O8 - O)) <= 1e-15
    assert np.allclose(LSE, math.log(2.0) * (-a.min()) + np.log(np.sum(2.0 ** -(a - a.min()))))


PINS = [pin_round_matches_torch, pin_saturation_and_codes, pin_fwht_is_sylvester, pin_quantize_round_trip,
        pin_fp8_forward_exact_parts, pin_fp8_power_of_two_probabilities]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_fp8_pin(pin):
    pin(fp8)


# ---------------------------------------------------------------------------
# Planted mistakes: each must fail at least one pin
# ---------------------------------------------------------------------------


def _mutant(name):
    m = types.ModuleType("fp8_mutant_" + name)
    m.__dict__.update({k: v for k, v in fp8.__dict__.items() if not k.startswith("__")})
    if name == "ties_away":
        def e4m3_round(x):
            x = np.asarray(x, dtype=np.float64)
            a = np.abs(x)
            _, E = np.frexp(a)
            e = np.maximum(E - 1, -6)
            q = np.ldexp(1.0, (e - 3).astype(np.int64))
            r = np.floor(a / q + 0.5) * q
            return np.copysign(np.minimum(np.where(a == 0, 0.0, r), 448.0), x)
        m.e4m3_round = e4m3_round
    elif name == "no_saturation":
        base = fp8.e4m3_round
        m.e4m3_round = lambda x: np.where(np.abs(np.asarray(x, dtype=np.float64)) > 448,
                                          np.asarray(x, dtype=np.float64), base(x))
    elif name == "subnormal_spacing":
        def e4m3_round(x):
            x = np.asarray(x, dtype=np.float64)
            a = np.abs(x)
            _, E = np.frexp(a)
            e = E - 1
            q = np.ldexp(1.0, (e - 3).astype(np.int64))
            r = np.rint(a / q) * q
            return np.copysign(np.minimum(np.where(a == 0, 0.0, r), 448.0), x)
        m.e4m3_round = e4m3_round
    elif name == "rotation_unnormalised":
        m.incoherent_rotate_f32 = lambda x, seed: fp8.fwht_f32(np.asarray(x, np.float32)
                                                               * fp8.hadamard_signs(np.shape(x)[-1], seed))
    elif name == "fwht_sign_flipped":
        def fwht_f32(x):
            y = np.array(x, dtype=np.float32, copy=True)
            d = y.shape[-1]
            h = 1
            while h < d:
                y = y.reshape(y.shape[:-1] + (d // (2 * h), 2, h))
                a, b = y[..., 0, :].copy(), y[..., 1, :].copy()
                y[..., 0, :], y[..., 1, :] = a + b, b - a
                y = y.reshape(y.shape[:-3] + (d,))
                h *= 2
            return y
        m.fwht_f32 = fwht_f32
    elif name == "descale_inverted":
        base = fp8.fp8_quantize_ref
        def fp8_quantize_ref(x, hadamard_seed=None, transpose=False):
            c, ds = base(x, hadamard_seed, transpose)
            return c, (1.0 / ds).astype(np.float32)
        m.fp8_quantize_ref = fp8_quantize_ref
    elif name == "p_not_rounded":
        def attn(q8, k8, vt8, dq, dk, dv, scale, causal):
            O, LSE, O8, bound = fp8.attn_fwd_fp8_ref(q8, k8, vt8, dq, dk, dv, scale, causal)
            return O, LSE, O, bound
        m.attn_fwd_fp8_ref = attn
    else:
        raise KeyError(name)
    # functions defined in the module body look globals up in their own module:
    # rebind them to the mutant's namespace so the planted function is the one called
    for k, v in list(m.__dict__.items()):
        if isinstance(v, types.FunctionType) and v.__module__ == fp8.__name__:
            m.__dict__[k] = types.FunctionType(v.__code__, m.__dict__, v.__name__, v.__defaults__, v.__closure__)
    return m


MUTANTS = ["ties_away", "no_saturation", "subnormal_spacing", "rotation_unnormalised", "fwht_sign_flipped",
           "descale_inverted", "p_not_rounded"]


@pytest.mark.parametrize("name", MUTANTS)
def test_fp8_mutant_is_caught(name):
    m = _mutant(name)
    caught = []
    for pin in PINS:
        try:
            pin(m)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passes every pin"
