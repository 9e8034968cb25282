"""Checks that tie the float64 oracle to facts it does not compute itself.

Each ``pin_*`` takes the oracle module (``oracle.attention``) and raises
AssertionError when a fact fails. The pin tests run them on the real oracle;
the mutation tests run them on copies with a planted mistake and expect a
failure, which shows the pins are sharp enough to catch that class of error.

Facts used: values the pages print (``tests/golden``), closed forms, library
routines (scipy's softmax / logsumexp, torch's float64 SDPA) and brute force in
pure-Python loops on tiny shapes.
"""
from __future__ import annotations

import json
import math
import os
import random

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _logit_row(A, x, values):
    """Run the definition on one query row whose logits are exactly x
    (d_h = 1, q = 1, k = x, scale = 1 gives S = x exactly)."""
    x = np.asarray(x, dtype=np.float64)
    q = np.ones((1, 1, 1))
    k = x.reshape(1, -1, 1)
    v = np.asarray(values, dtype=np.float64)[None]
    O, LSE = A.attention_ref(q, k, v, scale=1.0, causal=False)
    return O[0, 0], LSE[0, 0]


# ---------------------------------------------------------------------------

def pin_worked_example(A):
    """Printed worked example: [3,1] then [5,2]."""
    g = golden("worked_example.json")
    tol = g["printed_abs_tol"]
    (b1, b2) = g["blocks"]
    ones = np.ones((2, 1))
    s1 = A.block_state(b1, ones)
    assert abs(s1[0] - g["after_block_1"]["m"]) < tol
    assert abs(s1[1] - g["after_block_1"]["l"]) < tol
    s12 = A.merge_states(s1, A.block_state(b2, ones))
    assert abs(s12[0] - g["after_block_2"]["m"]) < tol
    assert abs(s12[1] - g["after_block_2"]["l"]) < tol
    # The streaming form reports the same rescale for block 2.
    x = np.array(b1 + b2)
    _, lse, alphas = A.online_softmax_attention(x, np.ones((4, 1)), block=2)
    assert abs(alphas[1] - g["rescale"]) < tol
    # LSE = m + ln(l), natural log, from the definition.
    o, lse_def = _logit_row(A, x, np.ones((4, 1)))
    assert abs(lse_def - (g["after_block_2"]["m"] + math.log(g["direct_l"]))) < tol
    assert abs(lse - lse_def) < 1e-12
    assert abs(o[0] - 1.0) < 1e-12


def pin_max_jump_rescale(A):
    """Printed rescale e^-5 = 0.0067379 when the max jumps 3 -> 8 in block 3."""
    g = golden("max_jump_rescale.json")
    maxima = g["block_maxima"]
    x = []
    for mx in maxima:
        x += [mx, mx - 1.5]
    vals = np.random.default_rng(1).normal(size=(8, 3))
    o, lse, alphas = A.online_softmax_attention(np.array(x), vals, block=2)
    assert abs(alphas[2] - g["alpha_block_3"]) < g["alpha_printed_abs_tol"]
    assert round(1.0 / alphas[2]) == g["divides_state_by"]
    o_def, lse_def = _logit_row(A, x, vals)
    assert np.allclose(o, o_def, rtol=1e-13, atol=1e-13)
    assert abs(lse - lse_def) < 1e-13


def pin_online_vs_safe(A):
    """The pages' numerical check: one-pass recurrence equals the safe softmax
    (and scipy's softmax / logsumexp) on 8192 logits with a late outlier."""
    from scipy.special import logsumexp, softmax

    g = golden("online_vs_safe.json")
    rng = np.random.default_rng(g["seed"])
    x = rng.normal(0, g["sigma"], g["N"])
    x[g["outlier_index"]] = g["outlier_value"]
    v = rng.normal(0, 1, (g["N"], g["D"]))
    o_on, lse_on, _ = A.online_softmax_attention(x, v, block=g["block"])
    o_def, lse_def = _logit_row(A, x, v)
    ref = softmax(x) @ v
    np.testing.assert_allclose(o_on, ref, rtol=g["rtol"], atol=g["atol"])
    np.testing.assert_allclose(o_def, ref, rtol=g["rtol"], atol=g["atol"])
    assert abs(lse_on - logsumexp(x)) < 1e-12
    assert abs(lse_def - logsumexp(x)) < 1e-12


def _fold_orders(A, states):
    seq = states[0]
    for s in states[1:]:
        seq = A.merge_states(seq, s)
    rev = states[-1]
    for s in reversed(states[:-1]):
        rev = A.merge_states(s, rev)
    idx = list(range(len(states)))
    random.Random(7).shuffle(idx)
    shf = states[idx[0]]
    for i in idx[1:]:
        shf = A.merge_states(shf, states[i])
    layer = list(states)
    while len(layer) > 1:
        nxt = [A.merge_states(layer[i], layer[i + 1]) for i in range(0, len(layer) - 1, 2)]
        if len(layer) % 2:
            nxt.append(layer[-1])
        layer = nxt
    return {"sequential": seq, "reversed": rev, "shuffled": shf, "tree": layer[0]}


def pin_merge_order(A):
    """Merge-order invariance on 1,000 keys, score std 30, uneven blocks with
    one block of length 1 and one fully masked block."""
    from scipy.special import logsumexp, softmax

    g = golden("merge_order.json")
    rng = np.random.default_rng(3)
    n = g["keys"]
    x = rng.normal(0, g["score_sigma"], n)
    v = rng.normal(0, 1, (n, 16))
    # Uneven blocks: [0,1), [37,38) and [999,1000) have length 1.
    cuts = [0, 1, 37, 38, 200, 431, 700, 999, 1000]
    bounds = list(zip(cuts[:-1], cuts[1:]))
    masked = (431, 700)  # this block is fully masked
    keep = np.ones(n, dtype=bool)
    keep[masked[0]:masked[1]] = False
    states = []
    for lo, hi in bounds:
        xb = x[lo:hi].copy()
        if (lo, hi) == masked:
            xb[:] = -np.inf
        states.append(A.block_state(xb, v[lo:hi]))
    folds = _fold_orders(A, states)
    outs = {k: A.finalize_state(s) for k, s in folds.items()}
    ref_o = softmax(x[keep]) @ v[keep]
    ref_lse = logsumexp(x[keep])
    for name, (o, lse) in outs.items():
        assert np.max(np.abs(o - ref_o)) <= g["tolerance"], name
        assert abs(lse - ref_lse) <= g["tolerance"] * max(1.0, abs(ref_lse)), name
    base = outs["sequential"][0]
    for name, (o, _) in outs.items():
        assert np.max(np.abs(o - base)) <= g["tolerance"], name


def pin_empty_identity(A):
    """The empty state is the merge identity; both-empty stays empty without NaN;
    an all-masked row gives zero output and LSE = -inf."""
    d = 5
    rng = np.random.default_rng(4)
    s = A.block_state(rng.normal(size=6), rng.normal(size=(6, d)))
    e = A.empty_state(d)
    with np.errstate(all="raise"):
        for a, b in ((e, s), (s, e)):
            m, l, acc = A.merge_states(a, b)
            assert m == s[0] and l == s[1] and np.array_equal(acc, s[2])
        m, l, acc = A.merge_states(e, A.block_state(np.full(3, -np.inf), np.ones((3, d))))
        assert np.isneginf(m) and l == 0.0 and not np.any(acc)
        o, lse = A.finalize_state(e)
        assert not np.any(o) and np.isneginf(lse)
    # Definition with a zero-length row through the page table.
    q = rng.normal(size=(2, 2, d))
    kc = rng.normal(size=(4, 16, 1, d))
    vc = rng.normal(size=(4, 16, 1, d))
    table = np.array([[0, 1], [2, 3]], dtype=np.int32)
    O, LSE = A.decode_paged_ref(q, kc, vc, table, np.array([0, 20]), 0.5)
    assert not np.any(O[0]) and np.all(np.isneginf(LSE[0]))
    assert np.all(np.isfinite(LSE[1]))
    # The N-way reduce: no active split, or all splits empty.
    o_p = rng.normal(size=(3, 4, d))
    m_p = rng.normal(size=(3, 4))
    l_p = rng.random((3, 4)) + 1
    m_p[2, :] = -np.inf
    l_p[2, :] = 0.0
    O, LSE = A.merge_partials_ref(o_p, m_p, l_p, n_active=[0, 4, 4])
    assert not np.any(O[0]) and np.isneginf(LSE[0])
    assert not np.any(O[2]) and np.isneginf(LSE[2])
    O, LSE = A.merge_lse_pair_ref(np.ones((1, d)), np.array([-np.inf]),
                                  np.ones((1, d)), np.array([-np.inf]))
    assert not np.any(O) and np.isneginf(LSE[0])


def pin_closed_forms(A):
    """Single key: O = v, LSE = x. Equal logits: O = mean(V), LSE = x + ln n.
    One dominant logit (+1000): O = its value vector."""
    rng = np.random.default_rng(5)
    d = 8
    v = rng.normal(size=(1, d))
    o, lse = _logit_row(A, [2.5], v)
    assert np.allclose(o, v[0], rtol=0, atol=1e-15) and abs(lse - 2.5) < 1e-15
    n = 37
    V = rng.normal(size=(n, d))
    o, lse = _logit_row(A, np.full(n, -1.25), V)
    assert np.allclose(o, V.mean(axis=0), rtol=1e-13, atol=1e-14)
    assert abs(lse - (-1.25 + math.log(n))) < 1e-13
    x = rng.normal(size=n)
    x[23] += 1000.0
    o, lse = _logit_row(A, x, V)
    assert np.allclose(o, V[23], rtol=0, atol=1e-14)
    assert abs(lse - x[23]) < 1e-12
    # GQA broadcast closed form: every query head of a group sees its KV head.
    h, h_kv, T = 4, 2, 3
    q = np.zeros((h, T, d))  # zero queries: uniform weights over allowed keys
    k = rng.normal(size=(h_kv, T, d))
    vv = rng.normal(size=(h_kv, T, d))
    O, LSE = A.attention_ref(q, k, vv, scale=0.3, causal=True)
    for hq in range(h):
        for i in range(T):
            assert np.allclose(O[hq, i], vv[hq // 2, :i + 1].mean(axis=0), atol=1e-14)
            assert abs(LSE[hq, i] - math.log(i + 1)) < 1e-14


def _brute_attention(q, k, v, scale, causal):
    h, T, d = len(q), len(q[0]), len(q[0][0])
    h_kv = len(k)
    g = h // h_kv
    O = [[[0.0] * d for _ in range(T)] for _ in range(h)]
    L = [[0.0] * T for _ in range(h)]
    for hq in range(h):
        kv = hq // g
        for i in range(T):
            js = [j for j in range(len(k[kv])) if (not causal or j <= i)]
            xs = [scale * sum(q[hq][i][c] * k[kv][j][c] for c in range(d)) for j in js]
            mx = max(xs)
            es = [math.exp(x - mx) for x in xs]
            tot = sum(es)
            for c in range(d):
                O[hq][i][c] = sum(es[t] * v[kv][js[t]][c] for t in range(len(js))) / tot
            L[hq][i] = mx + math.log(tot)
    return np.array(O), np.array(L)


def pin_brute_force_prefill(A):
    """Vectorised definition equals pure-Python loops on tiny GQA shapes."""
    rng = np.random.default_rng(6)
    for (h, h_kv, T, d, causal) in [(4, 2, 7, 3, True), (4, 2, 5, 3, False),
                                    (3, 1, 4, 2, True), (2, 2, 6, 4, False), (1, 1, 1, 3, True)]:
        q = rng.normal(size=(h, T, d))
        k = rng.normal(size=(h_kv, T, d))
        v = rng.normal(size=(h_kv, T, d))
        O, L = A.attention_ref(q, k, v, scale=0.7, causal=causal)
        Ob, Lb = _brute_attention(q.tolist(), k.tolist(), v.tolist(), 0.7, causal)
        assert np.allclose(O, Ob, rtol=1e-12, atol=1e-12)
        assert np.allclose(L, Lb, rtol=1e-12, atol=1e-12)
        # The whole-layer form (prefix slices), in a shuffled head order.
        order = list(range(h))[::-1]
        Oh, Lh = A.attention_heads_ref(q, k, v, 0.7, causal, order)
        assert np.allclose(Oh, Ob[order], rtol=1e-12, atol=1e-12)
        assert np.allclose(Lh, Lb[order], rtol=1e-12, atol=1e-12)
        # Sampled rows agree with the full definition.
        heads = [0, h - 1, h // 2]
        rows = [T - 1, 0, T // 2]
        Os, Ls = A.attention_rows_ref(q, k, v, 0.7, causal, heads, rows)
        for i, (hh, rr) in enumerate(zip(heads, rows)):
            assert np.allclose(Os[i], Ob[hh, rr], atol=1e-12)
            assert abs(Ls[i] - Lb[hh, rr]) < 1e-12


def pin_brute_force_decode(A):
    """Paged decode definition equals pure-Python loops over the page table,
    for lengths that are empty, one key, and end before/at/after a page edge."""
    rng = np.random.default_rng(8)
    page, h, h_kv, d = 16, 4, 2, 3
    lens = [0, 1, 15, 16, 17, 40]
    need = [(s + page - 1) // page for s in lens]
    nblk = sum(need) + 2
    perm = rng.permutation(nblk)
    table = -np.ones((len(lens), max(need)), dtype=np.int32)
    off = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[off:off + n]
        off += n
    q = rng.normal(size=(len(lens), h, d))
    kc = rng.normal(size=(nblk, page, h_kv, d))
    vc = rng.normal(size=(nblk, page, h_kv, d))
    O, L = A.decode_paged_ref(q, kc, vc, table, lens, 0.4)
    for b, s in enumerate(lens):
        for hq in range(h):
            kv = hq // (h // h_kv)
            if s == 0:
                assert not np.any(O[b, hq]) and np.isneginf(L[b, hq])
                continue
            xs, vs = [], []
            for p in range(s):
                phys = int(table[b][p // page])
                xs.append(0.4 * sum(q[b, hq, c] * kc[phys, p % page, kv, c] for c in range(d)))
                vs.append(vc[phys, p % page, kv])
            mx = max(xs)
            es = [math.exp(x - mx) for x in xs]
            tot = sum(es)
            ob = [sum(es[t] * vs[t][c] for t in range(s)) / tot for c in range(d)]
            assert np.allclose(O[b, hq], ob, atol=1e-12)
            assert abs(L[b, hq] - (mx + math.log(tot))) < 1e-12


def pin_library_sdpa(A):
    """Definition equals torch's float64 scaled_dot_product_attention (K/V
    repeated per group) and torch.logsumexp over the masked logits."""
    import torch

    rng = np.random.default_rng(9)
    for causal in (True, False):
        h, h_kv, T, d = 8, 2, 48, 16
        q = rng.normal(size=(h, T, d))
        k = rng.normal(size=(h_kv, T, d)) * 2
        v = rng.normal(size=(h_kv, T, d))
        O, L = A.attention_ref(q, k, v, scale=0.25, causal=causal)
        tq, tk, tv = (torch.from_numpy(t) for t in (q, k, v))
        tk = tk.repeat_interleave(h // h_kv, dim=0)
        tv = tv.repeat_interleave(h // h_kv, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(
            tq[None], tk[None], tv[None], is_causal=causal, scale=0.25)[0]
        assert np.allclose(O, ref.numpy(), rtol=1e-11, atol=1e-11)
        logits = 0.25 * tq @ tk.transpose(1, 2)
        if causal:
            logits = logits.masked_fill(torch.ones(T, T, dtype=torch.bool).triu(1), float("-inf"))
        lse_t = torch.logsumexp(logits, dim=-1).numpy()
        assert np.allclose(L, lse_t, rtol=1e-12, atol=1e-12)
        Oh, Lh = A.attention_heads_ref(q, k, v, 0.25, causal, range(h), threads=2)
        assert np.allclose(Oh, ref.numpy(), rtol=1e-11, atol=1e-11)
        assert np.allclose(Lh, lse_t, rtol=1e-12, atol=1e-12)


def pin_merge_partials(A):
    """N-way reduce of per-chunk states equals the definition over all keys,
    whatever the chunking; ignores splits at or past n_active."""
    from scipy.special import logsumexp, softmax

    rng = np.random.default_rng(10)
    d, S = 12, 6
    rows = 4
    o_p = np.full((rows, S, d), np.nan)
    m_p = np.full((rows, S), np.nan)
    l_p = np.full((rows, S), np.nan)
    n_act = [6, 3, 1, 5]
    refs = []
    for r in range(rows):
        n = 50 + 17 * r
        x = rng.normal(0, 8, n)
        v = rng.normal(size=(n, d))
        cuts = np.sort(rng.choice(np.arange(1, n), n_act[r] - 1, replace=False)).tolist()
        for i, (lo, hi) in enumerate(zip([0] + cuts, cuts + [n])):
            m, l, a = A.block_state(x[lo:hi], v[lo:hi])
            o_p[r, i], m_p[r, i], l_p[r, i] = a, m, l
        refs.append((softmax(x) @ v, logsumexp(x)))
    O, L = A.merge_partials_ref(o_p, m_p, l_p, n_active=n_act)
    for r in range(rows):
        assert np.allclose(O[r], refs[r][0], rtol=1e-12, atol=1e-12)
        assert abs(L[r] - refs[r][1]) < 1e-12


def pin_merge_lse_pair(A):
    """Two disjoint key ranges, each normalised with its LSE, merge to the
    definition over the union."""
    rng = np.random.default_rng(11)
    h, h_kv, T, d = 4, 2, 40, 8
    q = rng.normal(size=(h, 1, d))
    k = rng.normal(size=(h_kv, T, d)) * 3
    v = rng.normal(size=(h_kv, T, d))
    O, L = A.attention_ref(q, k, v, 0.3)
    Oa, La = A.attention_ref(q, k[:, :13], v[:, :13], 0.3)
    Ob, Lb = A.attention_ref(q, k[:, 13:], v[:, 13:], 0.3)
    Om, Lm = A.merge_lse_pair_ref(Oa[:, 0], La[:, 0], Ob[:, 0], Lb[:, 0])
    assert np.allclose(Om, O[:, 0], rtol=1e-12, atol=1e-12)
    assert np.allclose(Lm, L[:, 0], rtol=1e-12, atol=1e-12)


def pin_paged_prefill(A):
    """Variable-length paged rows: a row whose queries cover all its keys is
    the square causal definition on the gathered keys; a one-query row is the
    paged decode; tiny rows equal pure-Python loops with the queries at the
    row's last key positions."""
    rng = np.random.default_rng(21)
    page, h, h_kv, d = 16, 4, 2, 3
    q_lens = [5, 1, 3, 20]
    s_lens = [5, 37, 18, 20]
    need = [(s + page - 1) // page for s in s_lens]
    nblk = sum(need) + 1
    perm = rng.permutation(nblk)
    table = -np.ones((len(s_lens), max(need)), dtype=np.int32)
    off = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[off:off + n]
        off += n
    cu = np.concatenate([[0], np.cumsum(q_lens)])
    q = rng.normal(size=(int(cu[-1]), h, d))
    kc = rng.normal(size=(nblk, page, h_kv, d))
    vc = rng.normal(size=(nblk, page, h_kv, d))
    scale = 0.45
    O, L = A.prefill_paged_ref(q, kc, vc, table, cu, s_lens, scale, causal=True)

    def gather(b):
        s = s_lens[b]
        phys = [int(table[b][p // page]) for p in range(s)]
        K = np.stack([kc[phys[p], p % page] for p in range(s)], axis=1)  # [h_kv, s, d]
        V = np.stack([vc[phys[p], p % page] for p in range(s)], axis=1)
        return K, V

    # row 0 and row 3: queries cover every key -> square causal attention
    for b in (0, 3):
        K, V = gather(b)
        Oq, Lq = A.attention_ref(q[cu[b]:cu[b + 1]].transpose(1, 0, 2), K, V, scale, causal=True)
        assert np.allclose(O[cu[b]:cu[b + 1]], Oq.transpose(1, 0, 2), atol=1e-12)
        assert np.allclose(L[cu[b]:cu[b + 1]], Lq.T, atol=1e-12)
    # row 1: one query -> the paged decode of that row over all 37 keys
    Od, Ld = A.decode_paged_ref(q[cu[1]:cu[2]], kc, vc, table[1:2], [s_lens[1]], scale)
    assert np.allclose(O[cu[1]], Od[0], atol=1e-12) and np.allclose(L[cu[1]], Ld[0], atol=1e-12)
    # row 2: brute force, 3 queries at key positions 15, 16, 17 of 18
    b, s, ql = 2, s_lens[2], q_lens[2]
    for i in range(ql):
        posi = s - ql + i
        for hq in range(h):
            kv = hq // (h // h_kv)
            xs, vs = [], []
            for p_ in range(posi + 1):
                phys = int(table[b][p_ // page])
                xs.append(scale * sum(q[cu[b] + i, hq, c] * kc[phys, p_ % page, kv, c] for c in range(d)))
                vs.append(vc[phys, p_ % page, kv])
            mx = max(xs)
            es = [math.exp(x - mx) for x in xs]
            tot = sum(es)
            ob = [sum(es[t] * vs[t][c] for t in range(len(xs))) / tot for c in range(d)]
            assert np.allclose(O[cu[b] + i, hq], ob, atol=1e-12)
            assert abs(L[cu[b] + i, hq] - (mx + math.log(tot))) < 1e-12
    # without the mask every query of a row sees all of its keys
    On, Ln = A.prefill_paged_ref(q, kc, vc, table, cu, s_lens, scale, causal=False)
    Od, Ld = A.decode_paged_ref(q[cu[2]:cu[2] + 1], kc, vc, table[2:3], [s_lens[2]], scale)
    assert np.allclose(On[cu[2]], Od[0], atol=1e-12) and np.allclose(Ln[cu[2]], Ld[0], atol=1e-12)


def pin_nonfinite_inputs(A):
    """IEEE arithmetic on the definition over the allowed keys: a NaN logit
    makes its row NaN; a NaN / inf in v_j[e] reaches column e of exactly the
    rows that attend key j and no other element; a masked key's NaN reaches
    nothing. The merges carry a NaN state in either argument order."""
    rng = np.random.default_rng(31)
    h, h_kv, T, d = 2, 1, 6, 4
    q = rng.normal(size=(h, T, d))
    k = rng.normal(size=(h_kv, T, d))
    v = rng.normal(size=(h_kv, T, d))
    O0, L0 = A.attention_ref(q, k, v, 0.5, causal=True)
    with np.errstate(invalid="ignore"):
        kn = k.copy()
        kn[0, 3, 1] = np.nan  # logit of key 3 is NaN for every query
        O, L = A.attention_ref(q, kn, v, 0.5, causal=True)
        assert np.all(np.isnan(O[:, 3:])) and np.all(np.isnan(L[:, 3:]))
        assert np.array_equal(O[:, :3], O0[:, :3]) and np.array_equal(L[:, :3], L0[:, :3])
        for val in (np.nan, np.inf, -np.inf):
            vn = v.copy()
            vn[0, 2, 1] = val  # rows 2.. attend key 2 (weight > 0), rows 0, 1 do not
            O, L = A.attention_ref(q, k, vn, 0.5, causal=True)
            col = O[:, 2:, 1]
            assert (np.all(np.isnan(col)) if np.isnan(val) else np.all(col == val))
            keep = np.ones(O.shape, bool)
            keep[:, 2:, 1] = False
            assert np.array_equal(O[keep], O0[keep]) and np.array_equal(L, L0)
        # the same through the whole-layer and paged forms
        Oh, Lh = A.attention_heads_ref(q, kn, v, 0.5, True, range(h))
        assert np.all(np.isnan(Oh[:, 3:])) and np.array_equal(Oh[:, :3], O0[:, :3])
        # merges: a NaN state is not an empty one, in either order
        e = A.empty_state(d)
        bad = (np.nan, 1.0, np.ones(d))
        for a, b in ((e, bad), (bad, e)):
            assert np.isnan(A.merge_states(a, b)[0])
        for la, lb in ((np.nan, -np.inf), (-np.inf, np.nan), (np.nan, 0.5)):
            Om, Lm = A.merge_lse_pair_ref(np.ones((1, d)), np.array([la]), np.ones((1, d)),
                                          np.array([lb]))
            assert np.all(np.isnan(Om)) and np.isnan(Lm[0])
        Op, Lp = A.merge_partials_ref(np.ones((1, 3, d)), np.array([[0.0, np.nan, 1.0]]),
                                      np.ones((1, 3)))
        assert np.all(np.isnan(Op)) and np.isnan(Lp[0])
        o, lse, _ = A.online_softmax_attention(np.array([-np.inf, np.nan, 1.0]), np.ones((3, d)), 1)
        assert np.all(np.isnan(o)) and np.isnan(lse)


ALL_PINS = [
    pin_worked_example,
    pin_max_jump_rescale,
    pin_online_vs_safe,
    pin_merge_order,
    pin_empty_identity,
    pin_closed_forms,
    pin_brute_force_prefill,
    pin_brute_force_decode,
    pin_library_sdpa,
    pin_merge_partials,
    pin_merge_lse_pair,
    pin_paged_prefill,
    pin_nonfinite_inputs,
]
