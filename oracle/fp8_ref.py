"""FP8 (e4m3) attention forward: the oracle side.

TEST INFRASTRUCTURE ONLY (imported by the tests, the smoke check and the
benchmark's CPU legs; never by the product path).

The pages say only that FlashAttention-3 runs the forward on FP8 tensor cores
and lowers the quantisation error with "incoherent processing"
([WHY-FAST] "为什么Flash Attention能将注意力计算提速数倍而不损失精度", section
"Flash Attention 3：拥抱Hopper架构", item 3).  Everything below is this
project's reading, written out so that it can be checked by eye:

* e4m3 is the OCP FP8 E4M3FN format: 1 sign, 4 exponent (bias 7) and 3
  mantissa bits, no infinities, largest finite 448, subnormals down to 2^-9.
  Conversion rounds to nearest, ties to even, and saturates to +-448 (the
  PTX ``cvt.rn.satfinite`` rule).
* Quantisation is per (batch, head): every element of the head is multiplied
  by s = 448 / amax (fp32) and rounded to e4m3; the dequantisation factor
  ("descale") is amax / 448 (1 for an all-zero head).  All of it is fp32
  arithmetic, so the codes are an exact function of the inputs.
* Incoherent processing: Q and K are rotated along d by the same orthogonal
  matrix R = diag(sigma) H_d / sqrt(d) (H_d the Sylvester-Hadamard matrix,
  sigma_c = +-1 random signs), which leaves Q K^T unchanged (R R^T = I) and
  spreads outliers over all d columns before quantisation.  sigma_c is bit
  (c mod 128) of the 128-bit Philox4x32-10 output for counter
  (c div 128, 0, 0, 0) under the key (seed mod 2^32, seed div 2^32).  The
  transform is the fast Walsh-Hadamard butterfly (a, b) -> (a + b, a - b)
  with strides 1, 2, 4, ..., d/2, in fp32, then a multiply by
  fp32(1 / sqrt(d)).
* The forward computes S = scale (dq Q8)(dk K8)^T in fp32, the running-max
  softmax, and rounds the unnormalised probabilities P~ = exp(S - m) to e4m3
  before O = (P~ V8) dv / l, l the fp32 sum of the unrounded P~.  LSE is the
  plain one of S.
"""
from __future__ import annotations

import math
from typing import Optional, Tuple

import numpy as np

from .attention_ref import philox4x32_10

E4M3_MAX = 448.0


# ---------------------------------------------------------------------------
# The e4m3 format
# ---------------------------------------------------------------------------

def e4m3_round(x) -> np.ndarray:
    """Nearest e4m3 value (ties to even, saturating to +-448) of float64 x."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, E = np.frexp(a)                       # a = f 2^E, f in [0.5, 1)
    e = np.maximum(E - 1, -6)                # binade exponent; subnormals share 2^-6's spacing
    quantum = np.ldexp(1.0, (e - 3).astype(np.int64))   # 3 mantissa bits
    r = np.rint(a / quantum) * quantum       # np.rint: round half to even
    r = np.where(a == 0, 0.0, r)
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, x)


def e4m3_decode(codes) -> np.ndarray:
    """float64 values of e4m3 byte codes (0x7F / 0xFF are NaN)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, (e - 7)))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


def e4m3_encode(x) -> np.ndarray:
    """Byte codes of e4m3_round(x) (x finite); -0 encodes as 0x80."""
    r = e4m3_round(x)
    a = np.abs(r)
    _, E = np.frexp(a)
    e = E - 1
    normal = a >= 2.0 ** -6
    ebits = np.where(normal, e + 7, 0)
    mbits = np.where(normal, np.rint((a / np.ldexp(1.0, e.astype(np.int64)) - 1.0) * 8.0),
                     np.rint(a / 2.0 ** -9))
    mbits = np.where(a == 0, 0, mbits)
    ebits = np.where(a == 0, 0, ebits)
    code = (ebits.astype(np.int64) << 3) | mbits.astype(np.int64)
    code = code | np.where(np.signbit(r), 0x80, 0)
    return code.astype(np.uint8)


# ---------------------------------------------------------------------------
# Incoherent processing
# ---------------------------------------------------------------------------

def hadamard_signs(d: int, seed: int) -> np.ndarray:
    """sigma_c = 1 - 2 * bit c of the Philox stream described above (float32 +-1)."""
    out = np.empty(d, dtype=np.float32)
    for blk in range((d + 127) // 128):
        words = philox4x32_10(blk, 0, 0, 0, seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
        bits = [(int(words[c // 32]) >> (c % 32)) & 1 for c in range(128)]
        for c in range(128):
            if 128 * blk + c < d:
                out[128 * blk + c] = 1.0 - 2.0 * bits[c]
    return out


def fwht_f32(x: np.ndarray) -> np.ndarray:
    """Unnormalised fast Walsh-Hadamard transform along the last axis, float32
    butterflies (a, b) -> (a + b, a - b) with strides 1, 2, 4, ...: x H_d."""
    y = np.array(x, dtype=np.float32, copy=True)
    d = y.shape[-1]
    assert d & (d - 1) == 0, "power-of-two length"
    h = 1
    while h < d:
        y = y.reshape(y.shape[:-1] + (d // (2 * h), 2, h))
        a = y[..., 0, :].copy()
        b = y[..., 1, :].copy()
        y[..., 0, :] = a + b
        y[..., 1, :] = a - b
        y = y.reshape(y.shape[:-3] + (d,))
        h *= 2
    return y


def incoherent_rotate_f32(x, seed: int) -> np.ndarray:
    """x diag(sigma) H_d / sqrt(d) in the fp32 steps described above."""
    x = np.asarray(x, dtype=np.float32)
    d = x.shape[-1]
    y = fwht_f32(x * hadamard_signs(d, seed))
    return (y * np.float32(1.0 / math.sqrt(d))).astype(np.float32)


# ---------------------------------------------------------------------------
# Quantisation
# ---------------------------------------------------------------------------

def fp8_quantize_ref(x, hadamard_seed: Optional[int] = None,
                     transpose: bool = False) -> Tuple[np.ndarray, np.ndarray]:
    """Per-(b, h) e4m3 codes of a [B, H, N, d] tensor (fp32 steps: optional
    rotation, amax, s = 448 / amax, round(x s)) and the descale amax / 448.
    transpose=True returns the codes as [B, H, d, N]."""
    x = np.asarray(x, dtype=np.float32)
    if hadamard_seed is not None:
        x = incoherent_rotate_f32(x, hadamard_seed)
    B, H = x.shape[:2]
    codes = np.empty(x.shape, dtype=np.uint8)
    descale = np.empty((B, H), dtype=np.float32)
    for b in range(B):
        for h in range(H):
            amax = np.float32(np.max(np.abs(x[b, h]))) if x[b, h].size else np.float32(0)
            if amax > 0:
                s = np.float32(E4M3_MAX) / amax
                descale[b, h] = amax / np.float32(E4M3_MAX)
            else:
                s = np.float32(1.0)
                descale[b, h] = np.float32(1.0)
            codes[b, h] = e4m3_encode((x[b, h] * s).astype(np.float32).astype(np.float64))
    if transpose:
        codes = np.ascontiguousarray(np.swapaxes(codes, -1, -2))
    return codes, descale


def fp8_dequantize(codes, descale) -> np.ndarray:
    """float64 values descale[b, h] * e4m3(codes[b, h])."""
    return e4m3_decode(codes) * np.asarray(descale, dtype=np.float64)[:, :, None, None]


# ---------------------------------------------------------------------------
# Forward with e4m3 probabilities, and its error bound
# ---------------------------------------------------------------------------

def attn_fwd_fp8_ref(q8, k8, vt8, dq, dk, dv, scale: float,
                     causal: bool) -> Tuple[np.ndarray, np.ndarray, np.ndarray, np.ndarray]:
    """Reference for the FP8 forward on codes q8, k8 [B, H, N, d], vt8
    [B, H, d, N] with descales dq, dk, dv [B, H].  Returns (O_exact, LSE,
    O_p8, bound), float64:
      O_exact  softmax(scale Q K^T) V on the dequantised inputs (no rounding);
      LSE      its log-sum-exp;
      O_p8     the same with P~ = exp(S - rowmax) rounded to e4m3 before P~ V
               (l stays the sum of the unrounded P~), the kernel's arithmetic;
      bound    sum_j max(2^-4 P~_ij, 2^-10) |V_jc| / l_i, which bounds
               |O_p8 - O_exact| elementwise: an e4m3 rounding moves a value by
               at most half a unit in the last place, 2^-4 of it in the normal
               range and 2^-10 among the subnormals; the kernel's own
               reference max can only be smaller than the row's maximum
               by design, making its P~ larger and its subnormal floor
               relatively smaller."""
    Q = fp8_dequantize(q8, dq)
    K = fp8_dequantize(k8, dk)
    V = np.swapaxes(fp8_dequantize(vt8, dv), -1, -2)
    B, H, N, d = Q.shape
    Nk = K.shape[2]
    O = np.zeros((B, H, N, V.shape[-1]))
    O8 = np.zeros_like(O)
    bound = np.zeros_like(O)
    LSE = np.zeros((B, H, N))
    rows = np.arange(N)
    for b in range(B):
        for h in range(H):
            S = scale * (Q[b, h] @ K[b, h].T)
            if causal:
                S = np.where(np.arange(Nk)[None, :] > rows[:, None], -np.inf, S)
            m = S.max(axis=1, keepdims=True)
            Pt = np.exp(S - m)
            l = Pt.sum(axis=1, keepdims=True)
            O[b, h] = (Pt @ V[b, h]) / l
            O8[b, h] = (e4m3_round(Pt) @ V[b, h]) / l
            err = np.where(Pt > 0, np.maximum(Pt * 2.0 ** -4, 2.0 ** -10), 0.0)
            bound[b, h] = (err @ np.abs(V[b, h])) / l
            LSE[b, h] = m[:, 0] + np.log(l[:, 0])
    return O, LSE, O8, bound
