"""Float64 CPU oracle: plain, slow, obviously correct attention.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT: only the tests, the smoke check
and the benchmark's CPU-baseline / reference legs may use it. It shares no code
with the CUDA path.

Sources (page title, then section):
  [NA]  "Naive attention and the online softmax" (book §3.1)
  [OSR] "The Online Softmax Recurrence"
  [DEC] "Decode attention: FlashDecoding, split-K, paged kernels" (book §3.3)
  [MRG] "Merge normalized attention without averaging tile outputs"

Readings taken where the pages are silent:
  * LSE is the natural log: LSE = m + ln(l)  ([NA] "The state that gets passed
    around is the log-sum-exp"; [OSR] "What it buys").
  * A row with no allowed key has output 0 and LSE = -inf ([MRG], last
    paragraph, which offers zero output as the extension; [DEC] reduce step
    returns 0 when the exp-sum is 0).
  * Causal masking for equal query and key lengths: key j is allowed for
    query i iff j <= i. For a paged row with fewer queries than keys, the
    queries are the last key positions (bottom-right alignment).
  * Inputs are upcast to float64 exactly as stored (bf16 / fp32 values).
  * Non-finite inputs follow IEEE arithmetic on the definition over each
    row's allowed keys ([NA] "The base case is a NaN factory" shows how a
    NaN, once made, spreads through the weighted sums): a NaN logit (a NaN
    in q or in an attended k) makes the row's output and LSE NaN; a NaN or
    +-inf in an attended v_j[e] makes column e of the output NaN or +-inf;
    keys a row does not attend (masked, or past its length) are excluded
    and never reach it. Every max below propagates NaN (numpy's max does;
    Python's built-in max would drop a NaN depending on argument order).
"""
from __future__ import annotations

import math

import numpy as np

EMPTY_M = -np.inf


def _max_nan(a: float, b: float) -> float:
    """max(a, b), NaN if either is NaN."""
    if math.isnan(a) or math.isnan(b):
        return math.nan
    return max(a, b)


def to_f64(x) -> np.ndarray:
    """Upcast a numpy array or a (CPU) torch tensor to float64, value-exactly."""
    if hasattr(x, "detach"):
        x = x.detach().cpu()
        if str(x.dtype) in ("torch.bfloat16", "torch.float16"):
            x = x.float()
        x = x.numpy()
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# The definition: materialised safe softmax.
# ---------------------------------------------------------------------------

def _softmax_rows_times_v(S: np.ndarray, allowed: np.ndarray, V: np.ndarray):
    """Safe softmax of each row of S over its allowed entries, then times V.

    [NA] §(2) "Safe softmax": subtract the row maximum before exponentiating,
    which leaves the quotient unchanged (translation property of exp).
    Three passes: max, then sum of shifted exponentials, then normalise.
    Masked entries are excluded by index, never by a large negative number
    ([MRG]: masked logits are exclusions).
    Returns (O [n, d], LSE [n]).
    """
    n = S.shape[0]
    d = V.shape[1]
    O = np.zeros((n, d), dtype=np.float64)
    LSE = np.full(n, EMPTY_M, dtype=np.float64)
    for i in range(n):
        cols = np.nonzero(allowed[i])[0]
        if cols.size == 0:
            continue  # all-masked row: zero output, LSE = -inf ([MRG])
        x = S[i, cols]
        M = x.max()                      # pass 1: max
        p = np.exp(x - M)                # pass 2: shifted exponentials
        ell = p.sum()                    #          and their sum
        O[i] = (p / ell) @ V[cols]       # pass 3: normalise, weight the values
        LSE[i] = M + math.log(ell)       # LSE = m + ln(l)
    return O, LSE


def attention_ref(q, k, v, scale: float, causal: bool = False):
    """Exact scaled dot-product attention with grouped KV heads.

    [NA] opening section: Q is [h, T, d_h]; K and V are [h_kv, T, d_h] and are
    broadcast to the h/h_kv query heads of their group, so query head hq reads
    KV head hq // (h / h_kv).  S = scale * Q K^T is materialised per head.

    Returns O [h, Tq, d_h] and LSE [h, Tq] in float64.
    """
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    h, Tq, _ = q.shape
    h_kv, Tk, _ = k.shape
    d = v.shape[2]  # value width (equal to d_h for every workload here)
    if h % h_kv:
        raise ValueError("h must be a multiple of h_kv")
    if causal and Tq != Tk:
        raise ValueError("causal masking is defined here for equal query/key lengths")
    g = h // h_kv
    O = np.zeros((h, Tq, d), dtype=np.float64)
    LSE = np.full((h, Tq), EMPTY_M, dtype=np.float64)
    if causal:
        allowed = np.arange(Tk)[None, :] <= np.arange(Tq)[:, None]
    else:
        allowed = np.ones((Tq, Tk), dtype=bool)
    for hq in range(h):
        kvh = hq // g
        S = scale * (q[hq] @ k[kvh].T)
        O[hq], LSE[hq] = _softmax_rows_times_v(S, allowed, v[kvh])
    return O, LSE


def attention_rows_ref(q, k, v, scale: float, causal: bool, heads, rows):
    """``attention_ref`` evaluated only at the query positions (heads[i], rows[i]).

    Each output row of the definition depends on its own query row alone, so
    this is the same computation restricted to a sample (used where the full
    layer is too large for the oracle). Returns O [n, d_h], LSE [n].
    """
    k64, v64 = to_f64(k), to_f64(v)
    h = q.shape[0]
    h_kv, Tk, _ = k64.shape
    d = v64.shape[2]
    g = h // h_kv
    heads = np.asarray(heads, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    qsel = to_f64(q[heads, rows]) if hasattr(q, "detach") else to_f64(q)[heads, rows]
    O = np.zeros((len(rows), d), dtype=np.float64)
    LSE = np.full(len(rows), EMPTY_M, dtype=np.float64)
    for i, (hq, r) in enumerate(zip(heads.tolist(), rows.tolist())):
        kvh = hq // g
        S = scale * (qsel[i:i + 1] @ k64[kvh].T)
        allowed = np.ones((1, Tk), dtype=bool)
        if causal:
            allowed[0, r + 1:] = False
        O[i:i + 1], LSE[i:i + 1] = _softmax_rows_times_v(S, allowed, v64[kvh])
    return O, LSE


def _softmax_prefix_rows_times_v(S: np.ndarray, n_allowed, V: np.ndarray):
    """``_softmax_rows_times_v`` for rows whose allowed keys form a prefix.

    Row i may attend keys 0 .. n_allowed[i]-1: the causal rule j <= i gives
    n_allowed[i] = i + 1, and no mask gives every key. The allowed set is then
    a slice of S and V, so no index array is built and nothing is copied; the
    three passes ([NA] §(2) "Safe softmax") are those of
    ``_softmax_rows_times_v``. A row with no allowed key has zero output and
    LSE = -inf ([MRG]). Returns (O [n, d], LSE [n]).
    """
    n = S.shape[0]
    d = V.shape[1]
    O = np.zeros((n, d), dtype=np.float64)
    LSE = np.full(n, EMPTY_M, dtype=np.float64)
    for i in range(n):
        c = int(n_allowed[i])
        if c == 0:
            continue  # all-masked row: zero output, LSE = -inf ([MRG])
        x = S[i, :c]
        M = x.max()                      # pass 1: max
        p = np.exp(x - M)                # pass 2: shifted exponentials
        ell = p.sum()                    #          and their sum
        O[i] = (p / ell) @ V[:c]         # pass 3: normalise, weight the values
        LSE[i] = M + math.log(ell)       # LSE = m + ln(l)
    return O, LSE


def attention_heads_ref(q, k, v, scale: float, causal: bool, heads, threads: int = 1):
    """``attention_ref`` for the listed query heads, every query row.

    The definition of [NA]'s opening section (query head hq reads KV head
    hq // (h / h_kv); S = scale * q K^T materialised per head) with each row's
    allowed keys taken as a prefix of the key axis (``_softmax_prefix_rows_times_v``),
    which is what equal query and key lengths give under the causal rule j <= i.
    This is the form a whole long layer is checked with: one head at a time,
    optionally several heads at once on ``threads`` host threads (each head is
    independent; numpy releases the interpreter lock inside its loops).

    Returns O [len(heads), T, d] and LSE [len(heads), T] in float64, in the
    order of ``heads``.
    """
    q64, k64, v64 = to_f64(q), to_f64(k), to_f64(v)
    h, Tq, _ = q64.shape
    h_kv, Tk, _ = k64.shape
    d = v64.shape[2]
    if h % h_kv:
        raise ValueError("h must be a multiple of h_kv")
    if causal and Tq != Tk:
        raise ValueError("causal masking is defined here for equal query/key lengths")
    g = h // h_kv
    heads = [int(x) for x in heads]
    n_allowed = np.arange(1, Tq + 1) if causal else np.full(Tq, Tk)
    O = np.zeros((len(heads), Tq, d), dtype=np.float64)
    LSE = np.full((len(heads), Tq), EMPTY_M, dtype=np.float64)

    def one(idx):
        hq = heads[idx]
        kvh = hq // g
        S = scale * (q64[hq] @ k64[kvh].T)
        O[idx], LSE[idx] = _softmax_prefix_rows_times_v(S, n_allowed, v64[kvh])

    if threads <= 1:
        for idx in range(len(heads)):
            one(idx)
    else:
        from concurrent.futures import ThreadPoolExecutor

        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(one, range(len(heads))))
    return O, LSE


def decode_paged_ref(q, k_cache, v_cache, block_table, seq_lens, scale: float, rows=None):
    """One query token per row attending to its row's keys through a page table.

    [DEC] paged addressing: logical key position p of row b lives in physical
    page block_table[b][p // page_size] at slot p % page_size; the cache is
    laid out [page, slot, kv_head, d_h].  The keys 0 .. seq_len-1 are gathered
    into a contiguous [h_kv, s, d_h] block (upcast after gathering, so a large
    pool is never widened as a whole), then the definition is applied.
    A row with seq_len 0 has no keys: zero output, LSE = -inf.

    q [B, h, d_h] -> O [B, h, d_h], LSE [B, h] (float64). With ``rows`` only
    those rows are evaluated (the others stay 0 / -inf).
    """
    q64 = to_f64(q)
    table = np.asarray(block_table.cpu() if hasattr(block_table, "cpu") else block_table)
    lens = np.asarray(seq_lens.cpu() if hasattr(seq_lens, "cpu") else seq_lens).tolist()
    B, h, _ = q64.shape
    d = v_cache.shape[3]
    page = k_cache.shape[1]
    O = np.zeros((B, h, d), dtype=np.float64)
    LSE = np.full((B, h), EMPTY_M, dtype=np.float64)
    for b in (range(B) if rows is None else rows):
        s = int(lens[b])
        if s == 0:
            continue
        pos = np.arange(s)
        phys = table[b, pos // page].astype(np.int64)
        slot = pos % page
        if hasattr(k_cache, "detach"):
            import torch  # the caches may be CPU torch tensors (bf16)

            ip, isl = torch.from_numpy(phys), torch.from_numpy(slot)
            K = to_f64(k_cache[ip, isl]).transpose(1, 0, 2)  # [h_kv, s, d]
            V = to_f64(v_cache[ip, isl]).transpose(1, 0, 2)
        else:
            K = to_f64(k_cache[phys, slot]).transpose(1, 0, 2)
            V = to_f64(v_cache[phys, slot]).transpose(1, 0, 2)
        o, lse = attention_ref(q64[b][:, None, :], K, V, scale, causal=False)
        O[b] = o[:, 0]
        LSE[b] = lse[:, 0]
    return O, LSE


def _gather_row(k_cache, v_cache, table_row, s: int):
    """Keys 0 .. s-1 of one row through its page table, as [h_kv, s, d] float64."""
    page = k_cache.shape[1]
    pos = np.arange(s)
    phys = np.asarray(table_row)[pos // page].astype(np.int64)
    slot = pos % page
    if hasattr(k_cache, "detach"):
        import torch  # the caches may be CPU torch tensors (bf16)

        ip, isl = torch.from_numpy(phys), torch.from_numpy(slot)
        return (to_f64(k_cache[ip, isl]).transpose(1, 0, 2), to_f64(v_cache[ip, isl]).transpose(1, 0, 2))
    return (to_f64(k_cache[phys, slot]).transpose(1, 0, 2), to_f64(v_cache[phys, slot]).transpose(1, 0, 2))


def prefill_paged_ref(q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens, scale: float,
                      causal: bool = True, tokens=None):
    """Variable-length query rows over a paged KV cache (chunked prefill).

    Row b owns query tokens cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 of the packed
    q [total_q, h, d_h] and keys 0 .. seq_lens[b]-1 of the cache, gathered as in
    ``decode_paged_ref`` ([DEC] paged addressing). Reading for unequal lengths:
    the row's q_len queries are its last q_len key positions, so query i sits
    at position seq_len - q_len + i and, with ``causal``, sees keys up to and
    including that position (without it, all seq_len keys). Each allowed set
    then goes through the definition (materialised safe softmax, per head with
    the GQA broadcast of ``attention_ref``).

    Returns O [total_q, h, d_h] and LSE [total_q, h] (float64). With ``tokens``
    only those query tokens are evaluated (the others stay 0 / -inf).
    """
    q64 = to_f64(q)
    table = np.asarray(block_table.cpu() if hasattr(block_table, "cpu") else block_table)
    cu = np.asarray(cu_seqlens_q.cpu() if hasattr(cu_seqlens_q, "cpu") else cu_seqlens_q).tolist()
    lens = np.asarray(seq_lens.cpu() if hasattr(seq_lens, "cpu") else seq_lens).tolist()
    total_q, h, _ = q64.shape
    h_kv = k_cache.shape[2]
    d = v_cache.shape[3]
    g = h // h_kv
    O = np.zeros((total_q, h, d), dtype=np.float64)
    LSE = np.full((total_q, h), EMPTY_M, dtype=np.float64)
    want = None if tokens is None else set(int(t) for t in tokens)
    for b in range(len(lens)):
        t0, t1, s = int(cu[b]), int(cu[b + 1]), int(lens[b])
        q_len = t1 - t0
        if q_len == 0:
            continue
        if s < q_len:
            raise ValueError("a row needs at least as many keys as queries")
        sel = [i for i in range(q_len) if want is None or t0 + i in want]
        if not sel:
            continue
        K, V = _gather_row(k_cache, v_cache, table[b], s)
        pos = s - q_len + np.asarray(sel)  # key position of each selected query
        if causal:
            allowed = np.arange(s)[None, :] <= pos[:, None]
        else:
            allowed = np.ones((len(sel), s), dtype=bool)
        for hq in range(h):
            kvh = hq // g
            S = scale * (q64[t0 + np.asarray(sel), hq] @ K[kvh].T)
            o, lse = _softmax_rows_times_v(S, allowed, V[kvh])
            O[t0 + np.asarray(sel), hq] = o
            LSE[t0 + np.asarray(sel), hq] = lse
    return O, LSE


# ---------------------------------------------------------------------------
# Partial states (m, l, a) and their merge.
# ---------------------------------------------------------------------------

def empty_state(d: int):
    """The identity of the merge: m = -inf, l = 0, a = 0 ([OSR] "The recurrence";
    [NA] base case of the proof: max of the empty set is -inf, empty sum is 0)."""
    return (EMPTY_M, 0.0, np.zeros(d, dtype=np.float64))


def block_state(x, values):
    """Partial state of one block of keys.

    [OSR] "The recurrence": m is the block's max logit, l = sum exp(x - m) and
    a = sum exp(x - m) v.  Logits equal to -inf are masked keys and contribute
    nothing; a block with no unmasked key is the empty state ([MRG]: a fully
    masked tile contributes no keys).
    """
    x = np.asarray(x, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    keep = ~np.isneginf(x)
    if not keep.any():
        return empty_state(values.shape[1])
    xs, vs = x[keep], values[keep]
    m = xs.max()
    p = np.exp(xs - m)
    return (m, p.sum(), p @ vs)


def merge_states(a, b):
    """Merge two partial states over disjoint key sets.

    [OSR] "The recurrence" (general form) and [MRG] paragraph 3: take the
    larger max as the new reference, multiply each side's mass and numerator
    by exp(old max - new max), add.  [MRG] paragraph 5 and [NA] "The base case
    is a NaN factory": when both sides are empty the new max is -inf and
    -inf - (-inf) is NaN, so that case branches to the empty state instead.
    """
    (ma, la, xa), (mb, lb, xb) = a, b
    m = _max_nan(ma, mb)
    if np.isneginf(m):
        return empty_state(len(xa))
    wa = math.exp(ma - m) if not np.isneginf(ma) else 0.0
    wb = math.exp(mb - m) if not np.isneginf(mb) else 0.0
    return (m, la * wa + lb * wb, xa * wa + xb * wb)


def finalize_state(state):
    """Divide once at the end: o = a / l, LSE = m + ln l ([NA] "Extending the
    recurrence to the output"; LSE per "The state that gets passed around").
    An empty state gives o = 0, LSE = -inf."""
    m, ell, acc = state
    if ell == 0.0:
        return np.zeros_like(acc), EMPTY_M
    return acc / ell, m + math.log(ell)


def online_softmax_attention(x, values, block: int):
    """The streaming recurrence over consecutive key blocks of width ``block``.

    [NA] §(3) "The online recurrence" with the output extension: start from
    m = -inf, l = 0, O~ = 0; for each block take m_new = max(m, block max),
    alpha = exp(m - m_new) (0 while m is still -inf), p = exp(x_block - m_new),
    l = alpha l + sum p, O~ = alpha O~ + p V_block; finally o = O~ / l.
    Returns (o, LSE, alphas) where alphas lists the rescale factor per block.
    """
    x = np.asarray(x, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    m, ell, acc = EMPTY_M, 0.0, np.zeros(values.shape[1], dtype=np.float64)
    alphas = []
    for j in range(0, x.shape[0], block):
        xb, vb = x[j:j + block], values[j:j + block]
        m_new = _max_nan(m, xb.max())
        if np.isneginf(m_new):
            # Nothing unmasked seen yet: exp(-inf - (-inf)) would be NaN, so
            # the block is skipped ([NA] "The base case is a NaN factory").
            alphas.append(1.0)
            continue
        alpha = math.exp(m - m_new) if np.isfinite(m) else 0.0
        p = np.exp(xb - m_new)
        ell = alpha * ell + p.sum()
        acc = alpha * acc + p @ vb
        m = m_new
        alphas.append(alpha)
    if ell == 0.0:
        return np.zeros_like(acc), EMPTY_M, alphas
    o = acc / ell
    return o, m + math.log(ell), alphas


def merge_partials_ref(o_part, m_part, l_part, n_active=None):
    """N-way reduce of split partial states, one output row per input row.

    [DEC] stage 2 of split-KV ("reduce_segments"): over the row's active
    splits take the overall max M, rescale each split's l_i and O~_i by
    exp(m_i - M), sum, divide once.  A row with no active split, or whose
    summed mass is 0, returns 0 output and LSE = -inf.

    o_part [rows, S, d], m_part / l_part [rows, S]; n_active [rows] or None
    (all S splits active). Returns O [rows, d], LSE [rows] (float64).
    """
    o = to_f64(o_part)
    m = to_f64(m_part)
    l = to_f64(l_part)
    rows, S, d = o.shape
    na = [S] * rows if n_active is None else [int(t) for t in np.asarray(
        n_active.cpu() if hasattr(n_active, "cpu") else n_active)]
    O = np.zeros((rows, d), dtype=np.float64)
    LSE = np.full(rows, EMPTY_M, dtype=np.float64)
    for r in range(rows):
        n = na[r]
        if n <= 0:
            continue
        mi = m[r, :n]
        M = mi.max()
        if np.isneginf(M):
            continue
        w = np.exp(mi - M)
        L = (w * l[r, :n]).sum()
        if L == 0.0:
            continue
        O[r] = (w[:, None] * o[r, :n]).sum(axis=0) / L
        LSE[r] = M + math.log(L)
    return O, LSE


def merge_lse_pair_ref(o_a, lse_a, o_b, lse_b):
    """Symmetric merge of two normalised results over disjoint key sets.

    [NA] "The state that gets passed around is the log-sum-exp": with
    M = max(LSE_a, LSE_b), weights w = exp(LSE - M) / sum; the merged output is
    the convex combination w_a O_a + w_b O_b (weights first, then multiply --
    "Scale first, then multiply") and LSE = ln(sum) + M.  Both sides empty
    (M = -inf) gives 0 output and LSE = -inf.  Row-wise over [rows, d].
    """
    oa, ob = to_f64(o_a), to_f64(o_b)
    la, lb = to_f64(lse_a), to_f64(lse_b)
    O = np.zeros_like(oa)
    LSE = np.full(la.shape, EMPTY_M, dtype=np.float64)
    for r in range(la.shape[0]):
        M = _max_nan(la[r], lb[r])
        if np.isneginf(M):
            continue
        ea = math.exp(la[r] - M) if not np.isneginf(la[r]) else 0.0
        eb = math.exp(lb[r] - M) if not np.isneginf(lb[r]) else 0.0
        tot = ea + eb
        O[r] = (ea / tot) * oa[r] + (eb / tot) * ob[r]
        LSE[r] = math.log(tot) + M
    return O, LSE
