"""attn_merge_states (CUDA) against the oracle's N-way reduce."""
import numpy as np
import pytest
import torch

import online_softmax_attn_gb300 as attn
import oracle
import workloads as W
from parity import check_lse, check_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from online_softmax_attn_gb300 import build

    build.build()


@pytest.mark.parametrize("S", [1, 16, 17, 132])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_merge_random_partials(S, d, out_dtype):
    rows = 75
    g = torch.Generator().manual_seed(S * 1000 + d)
    n_active = torch.randint(0, S + 1, (rows,), generator=g, dtype=torch.int32)
    n_active[0] = 0
    n_active[1] = S
    o_p, m_p, l_p = W.partial_inputs(rows, S, d, seed=S + d, n_active=n_active)
    O_ref, L_ref = oracle.merge_partials_ref(o_p, m_p, l_p, n_active)
    dev = "cuda"
    o, lse = attn.attn_merge_states(o_p.to(dev), m_p.to(dev), l_p.to(dev), n_active.to(dev),
                                    out_dtype=out_dtype)
    check_out(o, O_ref, out_dtype)
    check_lse(lse, L_ref)
    assert attn.attn_get_device_error() == 0


def test_merge_all_active_when_no_counts():
    rows, S, d = 40, 8, 128
    o_p, m_p, l_p = W.partial_inputs(rows, S, d, seed=3)
    O_ref, L_ref = oracle.merge_partials_ref(o_p, m_p, l_p)
    o, lse = attn.attn_merge_states(o_p.cuda(), m_p.cuda(), l_p.cuda(), None, out_dtype=torch.float32)
    check_out(o, O_ref, torch.float32)
    check_lse(lse, L_ref)


def test_merge_of_key_chunks_equals_attention():
    """Partials made from real key chunks merge to the definition over all keys."""
    rng = np.random.default_rng(5)
    rows, S, d = 16, 7, 128
    o_p = np.full((rows, S, d), np.nan, np.float32)
    m_p = np.full((rows, S), np.nan, np.float32)
    l_p = np.full((rows, S), np.nan, np.float32)
    refs = []
    for r in range(rows):
        n = 300 + 11 * r
        x = rng.normal(0, 6, n)
        v = rng.normal(size=(n, d))
        cuts = np.linspace(0, n, S + 1).astype(int)
        for i in range(S):
            m, l, a = oracle.block_state(x[cuts[i]:cuts[i + 1]], v[cuts[i]:cuts[i + 1]])
            o_p[r, i], m_p[r, i], l_p[r, i] = a, m, l
        refs.append(oracle.finalize_state(oracle.merge_states(
            oracle.block_state(x, v), oracle.empty_state(d))))
    O_ref = np.stack([o for o, _ in refs])
    L_ref = np.array([l for _, l in refs])
    o, lse = attn.attn_merge_states(torch.from_numpy(o_p).cuda(), torch.from_numpy(m_p).cuda(),
                                    torch.from_numpy(l_p).cuda(), out_dtype=torch.float32)
    # fp32 partials carry fp32 rounding of the oracle's values: 1e-4 holds.
    check_out(o, O_ref, torch.float32)
    check_lse(lse, L_ref)


def test_merge_empty_rows_give_zero_not_nan():
    rows, S, d = 4, 5, 128
    o_p = torch.randn(rows, S, d)
    m_p = torch.full((rows, S), float("-inf"))
    l_p = torch.zeros(rows, S)
    m_p[3, 2] = 1.0
    l_p[3, 2] = 2.0
    n_active = torch.tensor([0, 5, 3, 5], dtype=torch.int32)
    o, lse = attn.attn_merge_states(o_p.cuda(), m_p.cuda(), l_p.cuda(), n_active.cuda(),
                                    out_dtype=torch.float32)
    o, lse = o.cpu(), lse.cpu()
    assert torch.all(o[:3] == 0) and torch.all(torch.isneginf(lse[:3]))
    assert torch.allclose(o[3], o_p[3, 2] / 2.0, atol=1e-6)
    assert abs(lse[3].item() - (1.0 + np.log(2.0))) < 1e-6
