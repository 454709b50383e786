"""fp64 CPU oracle for exact scaled-dot-product attention (TEST INFRASTRUCTURE ONLY).

Only the test suite, the smoke check and the benchmark's CPU-baseline /
reference arm may import this module.  The product path (the CUDA library and
its Python binding) never calls it, and it shares no code with that path.

Sources, cited by page title and section:
  [TRITON-IO]  page "FlashAttention的Triton实现：IO-aware注意力机制底层原理"
  [WHY-FAST]   page "为什么Flash Attention能将注意力计算提速数倍而不损失精度"
  [KERNEL-101] page "GPU Kernel 入门：Triton / FlashAttention"

What it computes.  The method is *exact* attention: tiling plus online
softmax reaches the plain result, up to rounding order ([WHY-FAST] §"在线Softmax
技巧"; [KERNEL-101] §"FlashAttention 与在线 softmax：难点与解法").  So the
oracle for the GPU path is the plain definition, written out with N x N score
and probability matrices materialised, in float64, on the (bf16-rounded)
inputs upcast exactly:

  S = scale * Q K^T, causal: S_ij = -inf for key j > query i
  m_i = max_j S_ij,  l_i = sum_j exp(S_ij - m_i),  P = exp(S - m) / l
  O = P V,  LSE_i = m_i + ln l_i

([WHY-FAST] §"标准注意力机制的内存困局" for S, P, O; §"在线Softmax技巧" for the
max-shifted ("safe") softmax; [TRITON-IO] §"Safe Softmax 的数学推导".)

Readings where the pages are silent (listed in the design notes):
  * the softmax scale never appears on the pages; it is a caller argument;
  * "masking" is named but not defined; causal keeps key j <= query i;
  * the pages save m and l; the oracle returns LSE = m + ln l (natural log);
  * a row with no unmasked key gets O = 0 and LSE = -inf (never NaN).

The backward is not given on the pages beyond "recompute S and P from the
saved blocks" ([WHY-FAST] §"反向传播中的重计算策略"); the oracle derives it by
calculus from the definition above (see ``attn_bwd_ref``).

The module also carries the pages' streaming algorithms (scalar online
softmax, the blockwise (m, l, acc) update, the two-block merge and a tiled
forward in the outer-Q / inner-KV order).  They are not used for GPU parity;
the tests pin them against the plain definition and the pages' worked example.
"""
from __future__ import annotations

import math
from typing import Optional, Tuple

import numpy as np

NEG_INF = -np.inf


# ---------------------------------------------------------------------------
# Plain definition, one (b, h) slice at a time
# ---------------------------------------------------------------------------

def _scores(qh: np.ndarray, kh: np.ndarray, scale: float) -> np.ndarray:
    """S = scale * Q K^T for one head ([WHY-FAST] §"标准注意力机制的内存困局")."""
    return scale * (qh @ kh.T)


def _apply_causal(S: np.ndarray, rows: np.ndarray) -> np.ndarray:
    """Set S[r, j] = -inf where key j is after query rows[r] (causal reading)."""
    cols = np.arange(S.shape[1])
    S = S.copy()
    S[cols[None, :] > rows[:, None]] = NEG_INF
    return S


def _softmax_stats(S: np.ndarray) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Safe softmax of each row: (P, m, l) with P = exp(S - m) / l.

    [WHY-FAST] §"在线Softmax技巧" (max-shifted softmax); rows with no finite
    score get P = 0, m = -inf, l = 0.
    """
    m = S.max(axis=1)
    m_shift = np.where(np.isfinite(m), m, 0.0)
    E = np.exp(S - m_shift[:, None])
    l = E.sum(axis=1)
    with np.errstate(invalid="ignore", divide="ignore"):
        P = np.where(l[:, None] > 0, E / np.where(l > 0, l, 1.0)[:, None], 0.0)
    return P, m, l


def _lse(m: np.ndarray, l: np.ndarray) -> np.ndarray:
    """LSE = m + ln l, -inf for an empty row."""
    with np.errstate(divide="ignore"):
        return np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), NEG_INF)


def _as64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def attn_fwd_ref(q, k, v, scale: float, causal: bool) -> Tuple[np.ndarray, np.ndarray]:
    """O [B,H,N,d] and LSE [B,H,N] in float64 for inputs of shape [B,H,N,d].

    Materialises S and P per (b, h) and applies the plain definition above.
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, H, N, d = q.shape
    O = np.zeros((B, H, N, v.shape[-1]))
    LSE = np.zeros((B, H, N))
    rows = np.arange(N)
    for b in range(B):
        for h in range(H):
            S = _scores(q[b, h], k[b, h], scale)
            if causal:
                S = _apply_causal(S, rows)
            P, m, l = _softmax_stats(S)
            O[b, h] = P @ v[b, h]
            LSE[b, h] = _lse(m, l)
    return O, LSE


def attn_fwd_ref_rows(q, k, v, scale: float, causal: bool,
                      rows: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """The plain definition evaluated only at selected query rows.

    ``rows`` has shape [B, H, R] (query indices per head).  Returns O [B,H,R,d]
    and LSE [B,H,R]; each row is computed exactly as in ``attn_fwd_ref``.
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    rows = np.asarray(rows, dtype=np.int64)
    B, H, R = rows.shape
    O = np.zeros((B, H, R, v.shape[-1]))
    LSE = np.zeros((B, H, R))
    for b in range(B):
        for h in range(H):
            r = rows[b, h]
            S = _scores(q[b, h][r], k[b, h], scale)
            if causal:
                S = _apply_causal(S, r)
            P, m, l = _softmax_stats(S)
            O[b, h] = P @ v[b, h]
            LSE[b, h] = _lse(m, l)
    return O, LSE


def attn_fwd_ref_end_aligned(q, k, v, scale: float) -> Tuple[np.ndarray, np.ndarray]:
    """Causal attention of a query block against a longer (or shorter) key
    sequence: O [B,H,Nq,d] and LSE [B,H,Nq] for q [B,H,Nq,d], k, v [B,H,Nk,d].

    The pages define the causal mask only for equal lengths.  Reading used
    here (and by the library's causal split-KV): the block is the last Nq
    positions of the Nk-long sequence, so query i sits at position
    Nk - Nq + i and sees the keys up to it; Nq == Nk is the square mask, a
    query before position 0 sees no key (O = 0, LSE = -inf, as any empty row).
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, H, Nq, _ = q.shape
    Nk = k.shape[2]
    O = np.zeros((B, H, Nq, v.shape[-1]))
    LSE = np.zeros((B, H, Nq))
    pos = np.arange(Nq) + (Nk - Nq)
    for b in range(B):
        for h in range(H):
            S = _apply_causal(_scores(q[b, h], k[b, h], scale), pos)
            P, m, l = _softmax_stats(S)
            O[b, h] = P @ v[b, h]
            LSE[b, h] = _lse(m, l)
    return O, LSE


def _grad_v(P: np.ndarray, doh: np.ndarray) -> np.ndarray:
    """dV = P^T dO."""
    return P.T @ doh


def _grad_p(doh: np.ndarray, vh: np.ndarray) -> np.ndarray:
    """dP = dO V^T."""
    return doh @ vh.T


def _row_term(doh: np.ndarray, O: np.ndarray) -> np.ndarray:
    """D_i = sum_c dO_ic O_ic (equals sum_j P_ij dP_ij because O = P V)."""
    return (doh * O).sum(axis=1)


def _grad_s(P: np.ndarray, dP: np.ndarray, D: np.ndarray) -> np.ndarray:
    """dS = P o (dP - D 1^T): the softmax Jacobian applied row by row."""
    return P * (dP - D[:, None])


def _grad_q(dS: np.ndarray, kh: np.ndarray, scale: float) -> np.ndarray:
    """dQ = scale * dS K."""
    return scale * (dS @ kh)


def _grad_k(dS: np.ndarray, qh: np.ndarray, scale: float) -> np.ndarray:
    """dK = scale * dS^T Q."""
    return scale * (dS.T @ qh)


def attn_bwd_ref(q, k, v, do, scale: float, causal: bool
                 ) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """dQ, dK, dV (float64) of L = <dO, O> for O = attn(q, k, v).

    Derived by calculus from the definition (the pages only say that the
    backward recomputes S and P, [WHY-FAST] §"反向传播中的重计算策略"):
      dV = P^T dO
      dP = dO V^T
      D_i = sum_j P_ij dP_ij  (= sum_c dO_ic O_ic, because O = P V)
      dS = P o (dP - D 1^T)   (softmax Jacobian; masked entries have P = 0)
      dQ = scale * dS K,   dK = scale * dS^T Q
    P is recomputed from Q, K exactly as in the forward.
    """
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    B, H, N, d = q.shape
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    rows = np.arange(N)
    for b in range(B):
        for h in range(H):
            S = _scores(q[b, h], k[b, h], scale)
            if causal:
                S = _apply_causal(S, rows)
            P, _, _ = _softmax_stats(S)
            O = P @ v[b, h]
            dv[b, h] = _grad_v(P, do[b, h])
            dP = _grad_p(do[b, h], v[b, h])
            dS = _grad_s(P, dP, _row_term(do[b, h], O))
            dq[b, h] = _grad_q(dS, k[b, h], scale)
            dk[b, h] = _grad_k(dS, q[b, h], scale)
    return dq, dk, dv


def attn_bwd_ref_sampled(q, k, v, do, scale: float, causal: bool, rows: np.ndarray, cols: np.ndarray,
                         group: int = 1024) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """The gradients of ``attn_bwd_ref`` at selected entries, for long rows.

    ``rows`` [B, H, R] selects the query rows of dQ, ``cols`` [B, H, C] the key
    rows of dK and dV.  Returns dQ [B,H,R,d], dK [B,H,C,d], dV [B,H,C,d].

    The formulas are those of ``attn_bwd_ref``.  dQ_i needs only row i of P
    and dP.  dK_j and dV_j sum over every query row i (dV_j = sum_i P_ij dO_i,
    dK_j = scale sum_i dS_ij Q_i), and each term needs D_i and so the whole
    forward row i: all query rows are evaluated, ``group`` of them at a time
    so that no N x N matrix is held; the groups' contributions are added in
    float64.  Nothing else is reordered.
    """
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    B, H, N, d = q.shape
    dq = np.zeros((B, H, rows.shape[2], d))
    dk = np.zeros((B, H, cols.shape[2], d))
    dv = np.zeros((B, H, cols.shape[2], v.shape[-1]))
    for b in range(B):
        for h in range(H):
            qh, kh, vh, doh = q[b, h], k[b, h], v[b, h], do[b, h]
            # dQ at the selected rows: rows of P, dP and dS
            r = rows[b, h]
            S = _scores(qh[r], kh, scale)
            if causal:
                S = _apply_causal(S, r)
            P, _, _ = _softmax_stats(S)
            dS = _grad_s(P, _grad_p(doh[r], vh), _row_term(doh[r], P @ vh))
            dq[b, h] = _grad_q(dS, kh, scale)
            # dK, dV at the selected keys: every query row contributes
            c = cols[b, h]
            for g0 in range(0, N, group):
                g = np.arange(g0, min(N, g0 + group))
                S = _scores(qh[g], kh, scale)
                if causal:
                    S = _apply_causal(S, g)
                P, _, _ = _softmax_stats(S)
                D = _row_term(doh[g], P @ vh)
                Pc = P[:, c]
                dv[b, h] += _grad_v(Pc, doh[g])
                dSc = _grad_s(Pc, _grad_p(doh[g], vh[c]), D)
                dk[b, h] += _grad_k(dSc, qh[g], scale)
    return dq, dk, dv


def bwd_preprocess_ref(o, do) -> np.ndarray:
    """D_i = sum_c dO_ic * O_ic per row, float64 [B,H,N] (the backward's row term)."""
    return (_as64(o) * _as64(do)).sum(axis=-1)


# ---------------------------------------------------------------------------
# Dropout on the probabilities (the pages name it only as a fused step of the
# GPU kernels, [WHY-FAST] §"标准注意力机制的内存困局"; the RNG contract below is
# this project's reading, written out in full)
# ---------------------------------------------------------------------------
#
# Random numbers: Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel
# random numbers: as easy as 1, 2, 3", SC 2011), a counter-based generator:
# ten rounds of two 32 x 32 -> 64-bit products with the multipliers
# 0xD2511F53 and 0xCD9E8D57, the key bumped by the Weyl constants 0x9E3779B9
# and 0xBB67AE85 between rounds.  Key = (seed mod 2^32, seed div 2^32).
#
# One call covers a 4 x 4 block of (query i, key j) for head bh:
#   counter = (j div 4, i div 4, bh, offset);  output word (i mod 4), byte
#   (j mod 4) (byte 0 = least significant) is the element's uniform byte u.
# Dropout probability p is quantised to t = round(256 p) clamped to [0, 255];
# the element is kept when u >= t, and kept probabilities are scaled by
# 256 / (256 - t), so E[mask * scale] = 1.
#   O = (P o Mt) V with Mt = keep * 256 / (256 - t), P the plain softmax;
#   LSE is the plain one (dropout acts after normalisation).

_PHILOX_M = (0xD2511F53, 0xCD9E8D57)
_PHILOX_W = (0x9E3779B9, 0xBB67AE85)
_U32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox4x32-10 on uint32 counter words (arrays broadcast) and key words;
    returns the four uint32 output words (computed in uint64)."""
    c = [np.asarray(x, dtype=np.uint64) & _U32 for x in (c0, c1, c2, c3)]
    k0 = np.uint64(int(k0) & 0xFFFFFFFF)
    k1 = np.uint64(int(k1) & 0xFFFFFFFF)
    m0, m1 = np.uint64(_PHILOX_M[0]), np.uint64(_PHILOX_M[1])
    w0, w1 = np.uint64(_PHILOX_W[0]), np.uint64(_PHILOX_W[1])
    for r in range(10):
        if r:
            k0 = (k0 + w0) & _U32
            k1 = (k1 + w1) & _U32
        p0 = m0 * c[0]
        p1 = m1 * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & _U32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _U32
        c = [(hi1 ^ c[1] ^ k0) & _U32, lo1, (hi0 ^ c[3] ^ k1) & _U32, lo0]
    return c


def dropout_threshold(p: float) -> int:
    """t = round(256 p), clamped to [0, 255]."""
    return int(min(255, max(0, math.floor(256.0 * float(p) + 0.5))))


def dropout_keep(bh: int, Nq: int, Nk: int, p: float, seed: int, offset: int) -> np.ndarray:
    """Keep mask [Nq, Nk] (bool) of head bh under the contract above."""
    i = np.arange(Nq, dtype=np.uint64)[:, None]
    j = np.arange(Nk, dtype=np.uint64)[None, :]
    words = philox4x32_10(j >> np.uint64(2), i >> np.uint64(2), np.uint64(bh), np.uint64(offset),
                          seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    sub = (i & np.uint64(3)) + np.zeros_like(j)      # word index = i mod 4
    word = np.select([sub == 0, sub == 1, sub == 2, sub == 3], words)
    u = (word >> ((j & np.uint64(3)) * np.uint64(8))) & np.uint64(0xFF)
    return u >= np.uint64(dropout_threshold(p))


def dropout_scale(p: float) -> float:
    t = dropout_threshold(p)
    return 256.0 / (256.0 - t)


def attn_fwd_dropout_ref(q, k, v, scale: float, causal: bool, p: float, seed: int,
                         offset: int, head0: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """O = (P o Mt) V and the plain LSE, float64, [B,H,N,d] inputs.  The mask of
    slice [b, h] is that of head index head0 + b*H + h (head0 > 0 for one head
    cut out of a larger batch)."""
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, H, N, d = q.shape
    O = np.zeros((B, H, N, v.shape[-1]))
    LSE = np.zeros((B, H, N))
    rows = np.arange(N)
    mult = dropout_scale(p)
    for b in range(B):
        for h in range(H):
            S = _scores(q[b, h], k[b, h], scale)
            if causal:
                S = _apply_causal(S, rows)
            P, m, l = _softmax_stats(S)
            Mt = dropout_keep(head0 + b * H + h, N, k.shape[2], p, seed, offset) * mult
            O[b, h] = (P * Mt) @ v[b, h]
            LSE[b, h] = _lse(m, l)
    return O, LSE


def _grad_s_dropout(P: np.ndarray, Mt: np.ndarray, dP: np.ndarray, D: np.ndarray) -> np.ndarray:
    """dS = P o (Mt o dP - D 1^T): the softmax Jacobian applied to dL/dP = Mt o dP."""
    return P * (Mt * dP - D[:, None])


def attn_bwd_dropout_ref(q, k, v, do, scale: float, causal: bool, p: float, seed: int,
                         offset: int, head0: int = 0) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """dQ, dK, dV of L = <dO, O> for the dropout forward above (fixed mask):
      dV = (P o Mt)^T dO,  dP = dO V^T,  D_i = sum_c dO_ic O_ic (O with dropout),
      dS = P o (Mt o dP - D 1^T),  dQ = scale dS K,  dK = scale dS^T Q
    (the softmax Jacobian applied to dL/dP = Mt o dP, whose row sums against P
    are D because O = (P o Mt) V)."""
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    B, H, N, d = q.shape
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    rows = np.arange(N)
    mult = dropout_scale(p)
    for b in range(B):
        for h in range(H):
            S = _scores(q[b, h], k[b, h], scale)
            if causal:
                S = _apply_causal(S, rows)
            P, _, _ = _softmax_stats(S)
            Mt = dropout_keep(head0 + b * H + h, N, k.shape[2], p, seed, offset) * mult
            Pd = P * Mt
            O = Pd @ v[b, h]
            dv[b, h] = Pd.T @ do[b, h]
            dP = _grad_p(do[b, h], v[b, h])
            dS = _grad_s_dropout(P, Mt, dP, _row_term(do[b, h], O))
            dq[b, h] = _grad_q(dS, k[b, h], scale)
            dk[b, h] = _grad_k(dS, q[b, h], scale)
    return dq, dk, dv


# ---------------------------------------------------------------------------
# The pages' streaming algorithms (pinned, not used for GPU parity)
# ---------------------------------------------------------------------------

def online_softmax_scalar(x) -> Tuple[float, float]:
    """Running (m, l) over a row, one element at a time.

    [TRITON-IO] §"Safe Softmax 的数学推导": on a new element x_{j+1},
    m_{j+1} = max(m_j, x_{j+1}) and l_{j+1} = l_j e^{m_j - m_{j+1}} + e^{x_{j+1} - m_{j+1}}.
    Starts from m = -inf, l = 0.
    """
    m, l = -math.inf, 0.0
    for xj in np.asarray(x, dtype=np.float64).ravel():
        m_new = max(m, float(xj))
        if m_new == -math.inf:
            continue
        l = l * math.exp(m - m_new) + math.exp(float(xj) - m_new)
        m = m_new
    return m, l


def online_softmax_blocks(scores, values, block: int) -> np.ndarray:
    """Softmax(scores) @ values streamed over key blocks with running (m, l, acc).

    [KERNEL-101] §"FlashAttention 与在线 softmax：难点与解法" and its hands-on
    section: per block, the new row max m_new = max(m, rowmax(block)); the old
    l and acc are scaled by e^{m - m_new}; the block adds sum e^{s - m_new} to l
    and e^{s - m_new} @ V_block to acc; at the end the result is acc / l.
    With ``values`` the identity this returns the softmax matrix itself.
    """
    s = _as64(scores)
    vals = _as64(values)
    R, C = s.shape
    m = np.full(R, NEG_INF)
    l = np.zeros(R)
    acc = np.zeros((R, vals.shape[1]))
    for c0 in range(0, C, block):
        blk = s[:, c0:c0 + block]
        m_new = np.maximum(m, blk.max(axis=1))
        safe_new = np.where(np.isfinite(m_new), m_new, 0.0)
        corr = np.where(np.isfinite(m), np.exp(m - safe_new), 0.0)
        e = np.exp(blk - safe_new[:, None])
        l = l * corr + e.sum(axis=1)
        acc = acc * corr[:, None] + e @ vals[c0:c0 + block]
        m = m_new
    with np.errstate(invalid="ignore", divide="ignore"):
        return np.where(l[:, None] > 0, acc / np.where(l > 0, l, 1.0)[:, None], 0.0)


def merge_two_blocks(m1, l1, o1, m2, l2, o2):
    """Combine the statistics of two key blocks of the same rows.

    [WHY-FAST] §"在线Softmax技巧": with m = max(m1, m2),
    l = e^{m1 - m} l1 + e^{m2 - m} l2 and the normalised outputs combine as
    O = (e^{m1 - m} l1 O1 + e^{m2 - m} l2 O2) / l.
    ``o1``/``o2`` are each block's own normalised output (rows x d).
    """
    m1, l1, o1, m2, l2, o2 = map(_as64, (m1, l1, o1, m2, l2, o2))
    m = np.maximum(m1, m2)
    safe = np.where(np.isfinite(m), m, 0.0)
    a1 = np.where(np.isfinite(m1), np.exp(m1 - safe), 0.0) * l1
    a2 = np.where(np.isfinite(m2), np.exp(m2 - safe), 0.0) * l2
    l = a1 + a2
    with np.errstate(invalid="ignore", divide="ignore"):
        o = np.where(l[:, None] > 0,
                     (a1[:, None] * o1 + a2[:, None] * o2) / np.where(l > 0, l, 1.0)[:, None],
                     0.0)
    return m, l, o


def attn_fwd_tiled_ref(q, k, v, scale: float, causal: bool, block_m: int = 64,
                       block_n: int = 64) -> Tuple[np.ndarray, np.ndarray]:
    """The tiled forward: outer loop over query tiles, inner loop over key tiles.

    Loop order of [TRITON-IO] §"FA1 vs FA2：循环顺序的工程权衡" (query tile
    outside, key/value tiles inside, accumulator kept for the whole inner loop),
    with the per-tile update of [WHY-FAST] §"分块计算（Tiling）" read in its
    consistent form (the new block's term is taken relative to the new max, the
    division by l happens once at the end, as in [KERNEL-101]'s hands-on
    section).  No N x N matrix is formed; float64 throughout.
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, H, N, d = q.shape
    Nk = k.shape[2]
    O = np.zeros((B, H, N, v.shape[-1]))
    LSE = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            for i0 in range(0, N, block_m):
                qi = q[b, h, i0:i0 + block_m]
                rows = np.arange(i0, i0 + qi.shape[0])
                m = np.full(qi.shape[0], NEG_INF)
                l = np.zeros(qi.shape[0])
                acc = np.zeros((qi.shape[0], v.shape[-1]))
                for j0 in range(0, Nk, block_n):
                    if causal and j0 > rows[-1]:
                        break
                    s = _scores(qi, k[b, h, j0:j0 + block_n], scale)
                    if causal:
                        cols = np.arange(j0, j0 + s.shape[1])
                        s = np.where(cols[None, :] > rows[:, None], NEG_INF, s)
                    m_new = np.maximum(m, s.max(axis=1))
                    safe_new = np.where(np.isfinite(m_new), m_new, 0.0)
                    corr = np.where(np.isfinite(m), np.exp(m - safe_new), 0.0)
                    p = np.exp(s - safe_new[:, None])
                    l = l * corr + p.sum(axis=1)
                    acc = acc * corr[:, None] + p @ v[b, h, j0:j0 + block_n]
                    m = m_new
                with np.errstate(invalid="ignore", divide="ignore"):
                    O[b, h, i0:i0 + block_m] = np.where(
                        l[:, None] > 0, acc / np.where(l > 0, l, 1.0)[:, None], 0.0)
                LSE[b, h, i0:i0 + block_m] = _lse(m, l)
    return O, LSE


# ---------------------------------------------------------------------------
# Error measures used by the parity tests
# ---------------------------------------------------------------------------

def max_abs_err(x, ref) -> float:
    x, ref = _as64(x), _as64(ref)
    if x.size == 0:
        return 0.0
    return float(np.max(np.abs(x - ref)))


def rel_fro_err(x, ref) -> float:
    x, ref = _as64(x), _as64(ref)
    den = float(np.linalg.norm(ref.ravel()))
    num = float(np.linalg.norm((x - ref).ravel()))
    return num / den if den > 0 else num


def lse_max_abs_err(x, ref) -> float:
    """Max |x - ref| over entries where ref is finite; -inf must match -inf."""
    x, ref = _as64(x), _as64(ref)
    fin = np.isfinite(ref)
    if np.any(~fin & (x != ref)):
        return math.inf
    if not np.any(fin):
        return 0.0
    return float(np.max(np.abs(x[fin] - ref[fin])))
