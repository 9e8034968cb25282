"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins
catch each one. A pin set that a dropped term, a wrong sign, a wrong index or a
transposed operand slips through would not be worth trusting."""
import math

import numpy as np
import pytest

import oracle.attention as A
import pins

_orig_attention_ref = A.attention_ref
_orig_softmax_rows = A._softmax_rows_times_v
_orig_softmax_prefix = A._softmax_prefix_rows_times_v


def _attention_variant(kv_of=None, allowed_of=None, swap_kv=False, drop_scale=False):
    def attention_ref(q, k, v, scale, causal=False):
        q, k, v = A.to_f64(q), A.to_f64(k), A.to_f64(v)
        if swap_kv and k.shape == v.shape:
            k, v = v, k
        h, Tq, _ = q.shape
        h_kv, Tk, _ = k.shape
        d = v.shape[2]
        g = h // h_kv
        O = np.zeros((h, Tq, d))
        L = np.full((h, Tq), -np.inf)
        allowed = (np.arange(Tk)[None, :] <= np.arange(Tq)[:, None]) if causal else np.ones((Tq, Tk), bool)
        if allowed_of is not None and causal:
            allowed = allowed_of(Tq, Tk)
        for hq in range(h):
            kvh = kv_of(hq, g, h_kv) if kv_of else hq // g
            S = (1.0 if drop_scale else scale) * (q[hq] @ k[kvh].T)
            O[hq], L[hq] = A._softmax_rows_times_v(S, allowed, v[kvh])
        return O, L
    return attention_ref


def _online_variant(rescale_acc=True, alpha_sign=1.0):
    def online(x, values, block):
        x = np.asarray(x, float)
        values = np.asarray(values, float)
        m, ell, acc = -np.inf, 0.0, np.zeros(values.shape[1])
        alphas = []
        for j in range(0, len(x), block):
            xb, vb = x[j:j + block], values[j:j + block]
            m_new = max(m, xb.max())
            alpha = math.exp(alpha_sign * (m - m_new)) if np.isfinite(m) else 0.0
            p = np.exp(xb - m_new)
            ell = alpha * ell + p.sum()
            acc = (alpha * acc if rescale_acc else acc) + p @ vb
            m = m_new
            alphas.append(alpha)
        return acc / ell, m + math.log(ell), alphas
    return online


def _merge_no_guard(a, b):
    (ma, la, xa), (mb, lb, xb) = a, b
    m = max(ma, mb)
    wa, wb = np.exp(ma - m), np.exp(mb - m)
    return (m, la * wa + lb * wb, xa * wa + xb * wb)


def _softmax_rows_log2(S, allowed, V):
    O, L = _orig_softmax_rows(S, allowed, V)
    M = np.array([S[i, allowed[i]].max() if allowed[i].any() else -np.inf for i in range(len(S))])
    return O, np.where(np.isfinite(L), M + (L - M) / math.log(2.0), L)


def _softmax_rows_no_shift_sum(S, allowed, V):
    # dropped term: the normaliser leaves out the first allowed key
    n, d = S.shape[0], V.shape[1]
    O = np.zeros((n, d))
    L = np.full(n, -np.inf)
    for i in range(n):
        cols = np.nonzero(allowed[i])[0]
        if cols.size == 0:
            continue
        x = S[i, cols]
        M = x.max()
        p = np.exp(x - M)
        ell = p[1:].sum() if p.size > 1 else p.sum()
        O[i] = (p / ell) @ V[cols]
        L[i] = M + math.log(ell)
    return O, L


def _softmax_prefix_drops_last(S, n_allowed, V):
    # wrong index: each row's prefix stops one key short (causal j < i)
    return _orig_softmax_prefix(S, [max(int(c) - 1, 1) for c in n_allowed], V)


def _merge_pair_drops_nan(o_a, lse_a, o_b, lse_b):
    # Python's max: max(-inf, nan) is -inf, so a NaN side can pass as empty
    oa, ob = A.to_f64(o_a), A.to_f64(o_b)
    la, lb = A.to_f64(lse_a), A.to_f64(lse_b)
    O = np.zeros_like(oa)
    L = np.full(la.shape, -np.inf)
    for r in range(la.shape[0]):
        M = max(la[r], lb[r])
        if np.isneginf(M):
            continue
        ea = math.exp(la[r] - M) if not np.isneginf(la[r]) else 0.0
        eb = math.exp(lb[r] - M) if not np.isneginf(lb[r]) else 0.0
        O[r] = (ea * oa[r] + eb * ob[r]) / (ea + eb)
        L[r] = math.log(ea + eb) + M
    return O, L


def _merge_partials_no_rescale(o_part, m_part, l_part, n_active=None):
    o, m, l = A.to_f64(o_part), A.to_f64(m_part), A.to_f64(l_part)
    rows, S, d = o.shape
    na = [S] * rows if n_active is None else list(n_active)
    O = np.zeros((rows, d))
    L = np.full(rows, -np.inf)
    for r in range(rows):
        n = int(na[r])
        if n <= 0:
            continue
        O[r] = o[r, :n].sum(0) / l[r, :n].sum()
        L[r] = m[r, :n].max() + math.log(l[r, :n].sum())
    return O, L


def _merge_pair_unweighted(o_a, lse_a, o_b, lse_b):
    oa, ob = A.to_f64(o_a), A.to_f64(o_b)
    la, lb = A.to_f64(lse_a), A.to_f64(lse_b)
    return 0.5 * (oa + ob), np.logaddexp(la, lb)


def _decode_slot_swapped(q, k_cache, v_cache, block_table, seq_lens, scale):
    q64, kc, vc = A.to_f64(q), A.to_f64(k_cache), A.to_f64(v_cache)
    table = np.asarray(block_table)
    B, h, _ = q64.shape
    page = kc.shape[1]
    O = np.zeros((B, h, vc.shape[3]))
    L = np.full((B, h), -np.inf)
    for b, s in enumerate(list(seq_lens)):
        s = int(s)
        if s == 0:
            continue
        pos = np.arange(s)
        phys = table[b, np.minimum(pos % page, table.shape[1] - 1)].astype(np.int64)
        phys = np.where(phys < 0, 0, phys)
        slot = np.minimum(pos // page, page - 1)
        K = kc[phys, slot].transpose(1, 0, 2)
        V = vc[phys, slot].transpose(1, 0, 2)
        o, lse = _orig_attention_ref(q64[b][:, None, :], K, V, scale)
        O[b], L[b] = o[:, 0], lse[:, 0]
    return O, L


def _paged_variant(top_left=False, ignore_mask=False):
    """prefill_paged_ref with the queries aligned to the first key positions,
    or with the causal mask ignored."""
    def prefill_paged_ref(q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens, scale,
                          causal=True, tokens=None):
        q64 = A.to_f64(q)
        table = np.asarray(block_table)
        cu = list(np.asarray(cu_seqlens_q))
        lens = list(np.asarray(seq_lens))
        total_q, h, _ = q64.shape
        h_kv = k_cache.shape[2]
        g = h // h_kv
        O = np.zeros((total_q, h, v_cache.shape[3]))
        L = np.full((total_q, h), -np.inf)
        for b in range(len(lens)):
            t0, t1, s_ = int(cu[b]), int(cu[b + 1]), int(lens[b])
            ql = t1 - t0
            if ql == 0:
                continue
            K, V = A._gather_row(k_cache, v_cache, table[b], s_)
            pos = np.arange(ql) if top_left else s_ - ql + np.arange(ql)
            allowed = (np.arange(s_)[None, :] <= pos[:, None]) if (causal and not ignore_mask) \
                else np.ones((ql, s_), bool)
            for hq in range(h):
                S = scale * (q64[t0:t1, hq] @ K[hq // g].T)
                O[t0:t1, hq], L[t0:t1, hq] = A._softmax_rows_times_v(S, allowed, V[hq // g])
        return O, L
    return prefill_paged_ref


MUTANTS = {
    # name: (attribute patches, pin expected to fail)
    "accumulator_not_rescaled": ({"online_softmax_attention": _online_variant(rescale_acc=False)},
                                 pins.pin_online_vs_safe),
    "alpha_sign_flipped": ({"online_softmax_attention": _online_variant(alpha_sign=-1.0)},
                           pins.pin_worked_example),
    "merge_without_empty_guard": ({"merge_states": _merge_no_guard}, pins.pin_empty_identity),
    "gqa_head_modulo": ({"attention_ref": _attention_variant(kv_of=lambda hq, g, hkv: hq % hkv)},
                        pins.pin_brute_force_prefill),
    "causal_strict_lower": ({"attention_ref": _attention_variant(
        allowed_of=lambda tq, tk: np.arange(tk)[None, :] < np.arange(tq)[:, None])},
        pins.pin_library_sdpa),
    "k_v_swapped": ({"attention_ref": _attention_variant(swap_kv=True)}, pins.pin_brute_force_prefill),
    "scale_dropped": ({"attention_ref": _attention_variant(drop_scale=True)}, pins.pin_library_sdpa),
    "lse_in_log2": ({"_softmax_rows_times_v": _softmax_rows_log2}, pins.pin_worked_example),
    "normaliser_term_dropped": ({"_softmax_rows_times_v": _softmax_rows_no_shift_sum},
                                pins.pin_closed_forms),
    "heads_prefix_one_short": ({"_softmax_prefix_rows_times_v": _softmax_prefix_drops_last},
                               pins.pin_brute_force_prefill),
    "split_partials_not_rescaled": ({"merge_partials_ref": _merge_partials_no_rescale},
                                    pins.pin_merge_partials),
    "pair_merge_unweighted": ({"merge_lse_pair_ref": _merge_pair_unweighted}, pins.pin_merge_lse_pair),
    "pair_merge_drops_nan": ({"merge_lse_pair_ref": _merge_pair_drops_nan}, pins.pin_nonfinite_inputs),
    "page_and_slot_swapped": ({"decode_paged_ref": _decode_slot_swapped}, pins.pin_brute_force_decode),
    "paged_queries_top_left": ({"prefill_paged_ref": _paged_variant(top_left=True)},
                               pins.pin_paged_prefill),
    "paged_mask_ignored": ({"prefill_paged_ref": _paged_variant(ignore_mask=True)},
                           pins.pin_paged_prefill),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pin_catches_mutant(name, monkeypatch):
    patches, pin = MUTANTS[name]
    for attr, fn in patches.items():
        monkeypatch.setattr(A, attr, fn)
    with pytest.raises((AssertionError, FloatingPointError, ValueError, IndexError)):
        with np.errstate(all="raise"):
            pin(A)


def test_unrescaled_accumulator_passes_when_max_is_first():
    """The failure the pages warn about: with the row max in the first block
    the missing accumulator rescale goes unnoticed (every later alpha is 1),
    which is why the pins put the max late."""
    x = np.concatenate([[50.0], np.random.default_rng(0).normal(size=255)])
    v = np.random.default_rng(1).normal(size=(256, 4))
    good, _, _ = A.online_softmax_attention(x, v, 64)
    bad, _, _ = _online_variant(rescale_acc=False)(x, v, 64)
    assert np.allclose(good, bad, rtol=1e-12, atol=1e-12)
