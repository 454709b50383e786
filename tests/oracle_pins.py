"""Pins for the fp64 oracle: facts fixed by the pages and by the mathematics.

Each ``pin_*`` takes an oracle module and raises AssertionError when the
oracle disagrees with something *other than itself*:
  * the pages' printed worked example (golden fixture, cited in the file);
  * closed forms (uniform scores, causal row 0, N = 1, a one-hot dominant key);
  * invariances (shifting keys or values, permuting key/value pairs, moving
    the scale between Q and the scale argument);
  * library routines for special cases (scipy's softmax / logsumexp);
  * central finite differences of L = <dO, O> for the backward, and the
    gradient identities sum_j dK_j = 0, sum_j dV_j = sum_i dO_i.

The same pins run against planted mistakes in ``test_oracle_mutants.py`` to
show that each plausible slip in the oracle is caught by at least one of them.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
from scipy import special

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return json.load(f)


def _rand(shape, seed, mult=1.0):
    return np.random.default_rng(seed).normal(size=shape) * mult


# ---------------------------------------------------------------------------
# Streaming algorithms (the pages' online softmax)
# ---------------------------------------------------------------------------

def pin_worked_example(ref):
    """Blockwise online softmax equals the whole-row softmax on the pages' case."""
    g = _golden("kernel101_online_softmax_worked_example.json")
    rng = np.random.default_rng(g["seed"])
    scores = rng.normal(size=tuple(g["shape"])) * g["multiplier"]
    whole = special.softmax(scores, axis=1)
    stream = ref.online_softmax_blocks(scores, np.eye(g["shape"][1]), g["block"])
    diff = float(np.abs(whole - stream).max())
    # The page prints 1.11e-16: float64 rounding, not bit-exact.  Same order.
    assert diff <= 4 * g["printed_max_abs_diff"], diff


def pin_online_scalar(ref):
    """Scalar running (m, l): m is the max and m + ln l the log-sum-exp."""
    for seed, n in [(1, 1), (2, 5), (3, 64), (4, 257)]:
        x = _rand(n, seed, 4.0)
        if n > 3:
            x[1] = -np.inf
        m, l = ref.online_softmax_scalar(x)
        assert m == np.max(x)
        assert abs((m + math.log(l)) - special.logsumexp(x)) <= 1e-13 * max(1.0, abs(m))


def pin_blockwise_random(ref):
    """Random rows, random block sizes, masked entries: equals softmax(S) @ V."""
    s = _rand((7, 37), 11, 5.0)
    s[2, 5:30] = -np.inf
    s[4, :36] = -np.inf
    v = _rand((37, 5), 12)
    want = special.softmax(s, axis=1) @ v
    for block in (1, 3, 8, 37, 50):
        got = ref.online_softmax_blocks(s, v, block)
        assert np.abs(got - want).max() <= 1e-13, block


def pin_merge(ref):
    """Two-block merge of (m, l, O), in any association order, equals the whole row."""
    s = _rand((6, 40), 21, 6.0)
    v = _rand((40, 3), 22)

    def stats(lo, hi):
        x = s[:, lo:hi]
        m = x.max(axis=1)
        l = np.exp(x - m[:, None]).sum(axis=1)
        o = special.softmax(x, axis=1) @ v[lo:hi]
        return m, l, o

    want_o = special.softmax(s, axis=1) @ v
    want_lse = special.logsumexp(s, axis=1)
    a, b, c = stats(0, 9), stats(9, 25), stats(25, 40)
    left = ref.merge_two_blocks(*ref.merge_two_blocks(*a, *b), *c)
    right = ref.merge_two_blocks(*a, *ref.merge_two_blocks(*b, *c))
    for m, l, o in (left, right):
        assert np.abs(o - want_o).max() <= 1e-13
        assert np.abs(m + np.log(l) - want_lse).max() <= 1e-12


def pin_tiled_equals_plain(ref):
    """The tiled outer-Q / inner-KV forward reaches the plain result (exactness)."""
    q, k, v = _rand((1, 2, 45, 6), 31), _rand((1, 2, 45, 6), 32), _rand((1, 2, 45, 6), 33)
    for causal in (False, True):
        o_ref, lse_ref = ref.attn_fwd_ref(q, k, v, 0.4, causal)
        for bm, bn in ((16, 16), (7, 13), (64, 64)):
            o, lse = ref.attn_fwd_tiled_ref(q, k, v, 0.4, causal, bm, bn)
            assert np.abs(o - o_ref).max() <= 1e-13
            assert np.abs(lse - lse_ref).max() <= 1e-12


# ---------------------------------------------------------------------------
# Forward definition: closed forms, special cases, invariances
# ---------------------------------------------------------------------------

def pin_library_softmax(ref):
    """Non-causal special case through scipy: O = softmax(sQK^T) V, LSE = logsumexp."""
    q, k, v = _rand((2, 1, 19, 4), 41), _rand((2, 1, 19, 4), 42), _rand((2, 1, 19, 4), 43)
    o, lse = ref.attn_fwd_ref(q, k, v, 0.3, False)
    for b in range(2):
        s = 0.3 * np.einsum("id,jd->ij", q[b, 0], k[b, 0])
        assert np.abs(o[b, 0] - special.softmax(s, axis=1) @ v[b, 0]).max() <= 1e-13
        assert np.abs(lse[b, 0] - special.logsumexp(s, axis=1)).max() <= 1e-12


def pin_uniform(ref):
    """Q = 0: every row is the mean of V (causal: of V[0..i]); LSE = ln(count)."""
    B, H, N, d = 2, 2, 37, 5
    q = np.zeros((B, H, N, d))
    k, v = _rand((B, H, N, d), 51), _rand((B, H, N, d), 52)
    o, lse = ref.attn_fwd_ref(q, k, v, 0.7, False)
    assert np.abs(o - v.mean(axis=2, keepdims=True)).max() <= 1e-13
    assert np.abs(lse - math.log(N)).max() <= 1e-13
    o, lse = ref.attn_fwd_ref(q, k, v, 0.7, True)
    counts = np.arange(1, N + 1)
    cum_mean = np.cumsum(v, axis=2) / counts[None, None, :, None]
    assert np.abs(o - cum_mean).max() <= 1e-13
    assert np.abs(lse - np.log(counts)[None, None, :]).max() <= 1e-13


def pin_one_hot(ref):
    """A key whose score leads all others by g returns its value row.

    With gap g, |O_i - V_j*| <= 2 (N-1) e^{-g} max|V| and
    0 <= LSE_i - s_ij* <= (N-1) e^{-g}.
    """
    N, d, scale = 33, 4, 0.5
    for causal in (False, True):
        for i in (0, 5, 32):
            jstar = (7 * i + 3) % (i + 1) if causal else (7 * i + 3) % N
            q = np.zeros((1, 1, N, d))
            q[0, 0, :, 0] = 1.0
            k = _rand((1, 1, N, d), 60 + i, 0.5)
            k[0, 0, jstar, 0] = 90.0           # s_ij* = 45, all others <= ~2
            v = _rand((1, 1, N, d), 70 + i)
            o, lse = ref.attn_fwd_ref(q, k, v, scale, causal)
            others = [j for j in range(N) if j != jstar and (not causal or j <= i)]
            s_star = scale * k[0, 0, jstar, 0]
            gap = s_star - max(scale * k[0, 0, j, 0] for j in others) if others else np.inf
            assert gap >= 40
            bound = 2 * (N - 1) * math.exp(-gap) * np.abs(v).max() + 1e-14
            assert np.abs(o[0, 0, i] - v[0, 0, jstar]).max() <= bound
            assert -1e-13 <= lse[0, 0, i] - s_star <= (N - 1) * math.exp(-gap) + 1e-13


def pin_causal_row0_and_n1(ref):
    """Causal row 0 sees only key 0: O_0 = V_0, LSE_0 = s q_0.k_0.  N = 1: O = V."""
    q, k, v = _rand((2, 3, 9, 4), 81), _rand((2, 3, 9, 4), 82), _rand((2, 3, 9, 4), 83)
    o, lse = ref.attn_fwd_ref(q, k, v, 0.6, True)
    assert np.abs(o[:, :, 0] - v[:, :, 0]).max() <= 1e-15
    dot0 = (q[:, :, 0] * k[:, :, 0]).sum(axis=-1)
    assert np.abs(lse[:, :, 0] - 0.6 * dot0).max() <= 1e-13
    for causal in (False, True):
        o1, lse1 = ref.attn_fwd_ref(q[:, :, :1], k[:, :, :1], v[:, :, :1], 0.6, causal)
        assert np.abs(o1 - v[:, :, :1]).max() <= 1e-15
        assert np.abs(lse1[:, :, 0] - 0.6 * dot0).max() <= 1e-13


def pin_invariances(ref):
    """Key shift, value shift, key/value permutation and scale placement."""
    B, H, N, d, s = 1, 2, 23, 6, 0.45
    q, k, v = _rand((B, H, N, d), 91), _rand((B, H, N, d), 92), _rand((B, H, N, d), 93)
    c = _rand(d, 94)
    for causal in (False, True):
        o, lse = ref.attn_fwd_ref(q, k, v, s, causal)
        # adding c to every key: O unchanged, LSE_i shifted by s q_i.c
        o2, lse2 = ref.attn_fwd_ref(q, k + c, v, s, causal)
        assert np.abs(o2 - o).max() <= 1e-12
        assert np.abs(lse2 - (lse + s * (q @ c))).max() <= 1e-12
        # adding c to every value: O shifted by c, LSE unchanged
        o3, lse3 = ref.attn_fwd_ref(q, k, v + c, s, causal)
        assert np.abs(o3 - (o + c)).max() <= 1e-12
        assert np.abs(lse3 - lse).max() <= 1e-13
        # the scale multiplies the scores: (2s, q/2) is the same problem
        o4, lse4 = ref.attn_fwd_ref(q / 2, k, v, 2 * s, causal)
        assert np.abs(o4 - o).max() <= 1e-12 and np.abs(lse4 - lse).max() <= 1e-12
    # permuting key/value pairs jointly leaves the non-causal result unchanged
    perm = np.random.default_rng(95).permutation(N)
    o, lse = ref.attn_fwd_ref(q, k, v, s, False)
    o5, lse5 = ref.attn_fwd_ref(q, k[:, :, perm], v[:, :, perm], s, False)
    assert np.abs(o5 - o).max() <= 1e-12 and np.abs(lse5 - lse).max() <= 1e-12
    # and a pure key permutation (without V) must change it
    o6, _ = ref.attn_fwd_ref(q, k[:, :, perm], v, s, False)
    assert np.abs(o6 - o).max() > 1e-3


def pin_rows_equals_full(ref):
    """The selected-rows evaluation equals the full evaluation at those rows."""
    q, k, v = _rand((2, 2, 50, 8), 101), _rand((2, 2, 50, 8), 102), _rand((2, 2, 50, 8), 103)
    rows = np.stack([np.stack([np.array([0, 3, 17, 49]), np.array([0, 1, 48, 49])])] * 2)
    for causal in (False, True):
        o, lse = ref.attn_fwd_ref(q, k, v, 0.35, causal)
        orr, lser = ref.attn_fwd_ref_rows(q, k, v, 0.35, causal, rows)
        for b in range(2):
            for h in range(2):
                assert np.abs(orr[b, h] - o[b, h, rows[b, h]]).max() <= 1e-14
                assert np.abs(lser[b, h] - lse[b, h, rows[b, h]]).max() <= 1e-14


# ---------------------------------------------------------------------------
# Backward
# ---------------------------------------------------------------------------

def _loss(ref, q, k, v, do, s, causal):
    o, _ = ref.attn_fwd_ref(q, k, v, s, causal)
    return float((o * do).sum())


def pin_finite_differences(ref):
    """Central differences of L = <dO, O> agree with the analytic gradients."""
    h = 1e-6
    for causal, (N, d), seed in ((False, (6, 3), 111), (True, (7, 4), 112), (False, (5, 2), 113)):
        q, k, v = (_rand((1, 1, N, d), seed + i) for i in range(3))
        do = _rand((1, 1, N, d), seed + 3)
        s = 0.7
        dq, dk, dv = ref.attn_bwd_ref(q, k, v, do, s, causal)
        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            fd = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = {"q": q, "k": k, "v": v}
                args_m = {"q": q, "k": k, "v": v}
                args_p[name], args_m[name] = xp, xm
                fd[idx] = (_loss(ref, args_p["q"], args_p["k"], args_p["v"], do, s, causal)
                           - _loss(ref, args_m["q"], args_m["k"], args_m["v"], do, s, causal)) / (2 * h)
            err = np.abs(fd - g).max() / max(1.0, np.abs(g).max())
            assert err <= 1e-7, (name, causal, err)


def pin_sampled_gradients(ref):
    """The sampled-entry backward (query rows taken in groups) agrees with
    central differences of L = <dO, O> at its entries, and with the
    materialised backward at every row and column."""
    h = 1e-6
    for causal, N, d, seed in ((False, 7, 3, 141), (True, 8, 2, 142)):
        q, k, v, do = (_rand((1, 1, N, d), seed + i) for i in range(4))
        s = 0.8
        rows = np.array([[[0, N - 1, 3]]])
        cols = np.array([[[N - 1, 0, 2]]])
        dq, dk, dv = ref.attn_bwd_ref_sampled(q, k, v, do, s, causal, rows, cols, group=3)
        for name, x, g, sel in (("q", q, dq, rows), ("k", k, dk, cols), ("v", v, dv, cols)):
            for a, r in enumerate(sel[0, 0]):
                for c in range(d):
                    xp, xm = x.copy(), x.copy()
                    xp[0, 0, r, c] += h
                    xm[0, 0, r, c] -= h
                    args_p = {"q": q, "k": k, "v": v}
                    args_m = {"q": q, "k": k, "v": v}
                    args_p[name], args_m[name] = xp, xm
                    fd = (_loss(ref, args_p["q"], args_p["k"], args_p["v"], do, s, causal)
                          - _loss(ref, args_m["q"], args_m["k"], args_m["v"], do, s, causal)) / (2 * h)
                    assert abs(fd - g[0, 0, a, c]) <= 1e-7 * max(1.0, abs(fd)), (name, causal, r, c)
    B, H, N, d = 2, 2, 50, 8
    q, k, v, do = (_rand((B, H, N, d), 150 + i) for i in range(4))
    every = np.broadcast_to(np.arange(N), (B, H, N))
    for causal in (False, True):
        full = ref.attn_bwd_ref(q, k, v, do, 0.45, causal)
        part = ref.attn_bwd_ref_sampled(q, k, v, do, 0.45, causal, every, every, group=16)
        for a, b in zip(full, part):
            assert np.abs(a - b).max() <= 1e-12 * max(1.0, np.abs(a).max())


def pin_gradient_identities(ref):
    """sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i; one-hot dO gives dV_j = P_ij g."""
    B, H, N, d, s = 1, 2, 21, 5, 0.5
    q, k, v, do = (_rand((B, H, N, d), 120 + i) for i in range(4))
    for causal in (False, True):
        dq, dk, dv = ref.attn_bwd_ref(q, k, v, do, s, causal)
        assert np.abs(dk.sum(axis=2)).max() <= 1e-12
        assert np.abs(dv.sum(axis=2) - do.sum(axis=2)).max() <= 1e-12
        # one-hot upstream gradient on row i: dV_j = P_ij * g, dQ, dK follow row i only
        i = 13
        g = _rand(d, 130)
        do1 = np.zeros_like(do)
        do1[:, :, i] = g
        _, _, dv1 = ref.attn_bwd_ref(q, k, v, do1, s, causal)
        _, lse = ref.attn_fwd_ref(q, k, v, s, causal)
        for h in range(H):
            srow = s * (k[0, h] @ q[0, h, i])
            if causal:
                srow[i + 1:] = -np.inf
            p = np.exp(srow - lse[0, h, i])
            assert abs(p.sum() - 1.0) <= 1e-12
            assert np.abs(dv1[0, h] - p[:, None] * g[None, :]).max() <= 1e-13


def pin_preprocess(ref):
    """D_i = sum_c dO_ic O_ic equals sum_j P_ij dP_ij with dP = dO V^T."""
    B, H, N, d, s = 1, 1, 17, 6, 0.6
    q, k, v, do = (_rand((B, H, N, d), 140 + i) for i in range(4))
    for causal in (False, True):
        o, lse = ref.attn_fwd_ref(q, k, v, s, causal)
        D = ref.bwd_preprocess_ref(o, do)
        S = s * (q[0, 0] @ k[0, 0].T)
        if causal:
            S[np.triu_indices(N, 1)] = -np.inf
        P = np.exp(S - lse[0, 0][:, None])
        dP = do[0, 0] @ v[0, 0].T
        assert np.abs(D[0, 0] - (P * dP).sum(axis=1)).max() <= 1e-12


def pin_unequal_lengths(ref):
    """Nq != Nk (short query blocks against long key sequences, non-causal):
    scipy's softmax / logsumexp per head, and with Q = 0 every row is the mean
    of all Nk values with LSE = ln Nk."""
    q, k, v = _rand((2, 2, 5, 4), 151), _rand((2, 2, 23, 4), 152), _rand((2, 2, 23, 4), 153)
    o, lse = ref.attn_fwd_ref(q, k, v, 0.45, False)
    assert o.shape == (2, 2, 5, 4) and lse.shape == (2, 2, 5)
    for b in range(2):
        for h in range(2):
            s = 0.45 * np.einsum("id,jd->ij", q[b, h], k[b, h])
            assert np.abs(o[b, h] - special.softmax(s, axis=1) @ v[b, h]).max() <= 1e-13
            assert np.abs(lse[b, h] - special.logsumexp(s, axis=1)).max() <= 1e-12
    o, lse = ref.attn_fwd_ref(np.zeros((1, 1, 3, 4)), k[:1, :1], v[:1, :1], 0.45, False)
    assert np.abs(o - v[:1, :1].mean(axis=2, keepdims=True)).max() <= 1e-13
    assert np.abs(lse - math.log(23)).max() <= 1e-13


def pin_causal_end_aligned(ref):
    """Causal blocks aligned to the end of the keys (query i at position
    Nk - Nq + i): Nq == Nk is the square causal mask; a block is the last Nq
    rows of the square problem; one row sees every key; with Q = 0 row i is
    the mean of V[0 .. Nk - Nq + i] with LSE = ln(Nk - Nq + i + 1); queries
    before position 0 are empty rows (O = 0, LSE = -inf)."""
    qf, k, v = _rand((2, 2, 23, 4), 161), _rand((2, 2, 23, 4), 162), _rand((2, 2, 23, 4), 163)
    o_sq, l_sq = ref.attn_fwd_ref(qf, k, v, 0.4, True)
    o, lse = ref.attn_fwd_ref_end_aligned(qf, k, v, 0.4)
    assert np.abs(o - o_sq).max() <= 1e-14 and np.abs(lse - l_sq).max() <= 1e-14
    o5, l5 = ref.attn_fwd_ref_end_aligned(qf[:, :, -5:], k, v, 0.4)
    assert np.abs(o5 - o_sq[:, :, -5:]).max() <= 1e-14 and np.abs(l5 - l_sq[:, :, -5:]).max() <= 1e-14
    o1, l1 = ref.attn_fwd_ref_end_aligned(qf[:, :, :1], k, v, 0.4)
    o1n, l1n = ref.attn_fwd_ref(qf[:, :, :1], k, v, 0.4, False)
    assert np.abs(o1 - o1n).max() <= 1e-14 and np.abs(l1 - l1n).max() <= 1e-14
    oz, lz = ref.attn_fwd_ref_end_aligned(np.zeros((1, 1, 6, 4)), k[:1, :1], v[:1, :1], 0.4)
    for i in range(6):
        n = 23 - 6 + i + 1
        assert np.abs(oz[0, 0, i] - v[0, 0, :n].mean(axis=0)).max() <= 1e-13
        assert abs(lz[0, 0, i] - math.log(n)) <= 1e-13
    q30 = _rand((1, 1, 30, 4), 164)
    o30, l30 = ref.attn_fwd_ref_end_aligned(q30, k[:1, :1], v[:1, :1], 0.4)
    assert np.all(o30[:, :, :7] == 0) and np.all(np.isneginf(l30[:, :, :7]))
    o23, l23 = ref.attn_fwd_ref(q30[:, :, 7:], k[:1, :1], v[:1, :1], 0.4, True)
    assert np.abs(o30[:, :, 7:] - o23).max() <= 1e-14 and np.abs(l30[:, :, 7:] - l23).max() <= 1e-14


# ---------------------------------------------------------------------------
# Dropout: the counter-based generator and the dropout algebra
# ---------------------------------------------------------------------------

def pin_philox_known_answers(ref):
    """Philox4x32-10 reproduces the generator's published known-answer vectors
    (counter, key -> output), from all-zero, all-ones and pi-digit inputs."""
    cases = [((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
             ((0xFFFFFFFF,) * 4, (0xFFFFFFFF, 0xFFFFFFFF), (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
             ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
              (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1))]
    for ctr, key, want in cases:
        got = tuple(int(x) for x in ref.philox4x32_10(*ctr, *key))
        assert got == want, [hex(x) for x in got]


def pin_dropout_p0_is_plain(ref):
    """Dropout probability 0 keeps everything with scale 1: the plain results."""
    q, k, v, do = (_rand((1, 2, 13, 4), 160 + i) for i in range(4))
    for causal in (False, True):
        o, lse = ref.attn_fwd_ref(q, k, v, 0.5, causal)
        od, lsed = ref.attn_fwd_dropout_ref(q, k, v, 0.5, causal, 0.0, 99, 3)
        assert np.abs(od - o).max() <= 1e-15 and np.abs(lsed - lse).max() <= 1e-15
        g = ref.attn_bwd_ref(q, k, v, do, 0.5, causal)
        gd = ref.attn_bwd_dropout_ref(q, k, v, do, 0.5, causal, 0.0, 99, 3)
        for a, b in zip(gd, g):
            assert np.abs(a - b).max() <= 1e-14


def pin_dropout_rates(ref):
    """Keep fractions match 1 - t/256 and the uniform bytes are flat (6-sigma bounds)."""
    for p in (0.1, 0.3, 0.5, 0.9):
        m = ref.dropout_keep(2, 200, 300, p, 0x0123456789ABCDEF, 11)
        keep = 1.0 - ref.dropout_threshold(p) / 256.0
        sd = math.sqrt(keep * (1 - keep) / m.size)
        assert abs(m.mean() - keep) <= 6 * sd, (p, m.mean(), keep)
    w = ref.philox4x32_10(np.arange(4096), 5, 6, 7, 0xDEADBEEF, 0x12345678)
    b = np.concatenate([(np.asarray(x, dtype=np.uint64) >> np.uint64(8 * s)) & np.uint64(0xFF)
                        for x in w for s in range(4)]).astype(np.int64)
    counts = np.bincount(b, minlength=256)
    e = b.size / 256.0
    chi2 = float(((counts - e) ** 2 / e).sum())
    assert chi2 <= 255 + 6 * math.sqrt(2 * 255), chi2


def pin_dropout_unbiased(ref):
    """Averaged over many masks (offsets) the output approaches the plain one:
    with V = 1 every plain row is exactly 1, and E[Mt] = 1 (variance <= 1 per mask)."""
    q, k = _rand((1, 1, 12, 3), 171), _rand((1, 1, 12, 3), 172)
    v = np.ones((1, 1, 12, 3))
    acc = np.zeros((1, 1, 12, 3))
    n = 400
    for off in range(n):
        acc += ref.attn_fwd_dropout_ref(q, k, v, 0.8, False, 0.5, 2024, off)[0]
    assert np.abs(acc / n - 1.0).max() <= 6 / math.sqrt(n)


def pin_dropout_finite_differences(ref):
    """Central differences of L = <dO, O> with the mask fixed agree with the dropout backward."""
    h = 1e-6
    for causal, (N, d), seed in ((False, (6, 3), 181), (True, (7, 4), 182)):
        q, k, v = (_rand((1, 1, N, d), seed + i) for i in range(3))
        do = _rand((1, 1, N, d), seed + 3)
        s, p, sd, off = 0.7, 0.3, 77, 5
        dq, dk, dv = ref.attn_bwd_dropout_ref(q, k, v, do, s, causal, p, sd, off)
        loss = lambda a, b, c: float((ref.attn_fwd_dropout_ref(a, b, c, s, causal, p, sd, off)[0] * do).sum())
        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            fd = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                ap = {"q": q, "k": k, "v": v}
                am = {"q": q, "k": k, "v": v}
                ap[name], am[name] = xp, xm
                fd[idx] = (loss(ap["q"], ap["k"], ap["v"]) - loss(am["q"], am["k"], am["v"])) / (2 * h)
            err = np.abs(fd - g).max() / max(1.0, np.abs(g).max())
            assert err <= 1e-7, (name, causal, err)


ALL_PINS = [
    pin_worked_example,
    pin_online_scalar,
    pin_blockwise_random,
    pin_merge,
    pin_tiled_equals_plain,
    pin_library_softmax,
    pin_uniform,
    pin_one_hot,
    pin_causal_row0_and_n1,
    pin_invariances,
    pin_rows_equals_full,
    pin_causal_end_aligned,
    pin_finite_differences,
    pin_sampled_gradients,
    pin_gradient_identities,
    pin_preprocess,
    pin_unequal_lengths,
    pin_philox_known_answers,
    pin_dropout_p0_is_plain,
    pin_dropout_rates,
    pin_dropout_unbiased,
    pin_dropout_finite_differences,
]
