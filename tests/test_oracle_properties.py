"""Property pins of the fp64 oracle's attention over random packed layouts (CPU only).

Each property holds exactly in the mathematics of per-segment softmax attention and
catches one family of index mistakes: a key permutation inside a segment leaves every
output unchanged (k and v rows paired wrongly), a query permutation permutes the outputs
(a wrong query-row offset), reordering whole segments in the packed stream moves their
outputs with them (a wrong segment offset), heads computed together equal heads computed
one at a time (head mixing), a scale folded into q changes nothing (a scale applied twice
or dropped), and the output is linear in v (k used for v). Layouts are drawn by
hypothesis, empty and one-token segments included, with a fixed seed for reproducibility."""
import numpy as np
import pytest

import oracle
from oracle.dense_ref import dense_block_diag_attention

hypothesis = pytest.importorskip("hypothesis")
st = hypothesis.strategies
given, settings = hypothesis.given, hypothesis.settings

TOL = 1e-12
layouts = st.lists(st.integers(0, 24), min_size=1, max_size=5)
_settings = settings(max_examples=40, deadline=None, derandomize=True)


def _inputs(lengths, H, D, seed):
    rng = np.random.default_rng(seed)
    T = int(sum(lengths))
    q, k, v = (rng.standard_normal((T, H, D)) for _ in range(3))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return q, k, v, cu


@_settings
@given(lengths=layouts, H=st.integers(1, 3), D=st.sampled_from([4, 8, 16]), seed=st.integers(0, 2 ** 16))
def test_dense_mask_form_equals_per_segment_form(lengths, H, D, seed):
    q, k, v, cu = _inputs(lengths, H, D, seed)
    if q.shape[0] == 0:
        return
    np.testing.assert_allclose(oracle.attention(q, k, v, cu), dense_block_diag_attention(q, k, v, cu),
                               rtol=0, atol=TOL)


@_settings
@given(lengths=layouts, H=st.integers(1, 3), D=st.sampled_from([4, 8]), seed=st.integers(0, 2 ** 16))
def test_key_and_query_permutations_inside_segments(lengths, H, D, seed):
    q, k, v, cu = _inputs(lengths, H, D, seed)
    base = oracle.attention(q, k, v, cu)
    rng = np.random.default_rng(seed + 1)
    pk = np.arange(q.shape[0])
    pq = np.arange(q.shape[0])
    for a, b in zip(cu[:-1], cu[1:]):
        pk[a:b] = a + rng.permutation(b - a)
        pq[a:b] = a + rng.permutation(b - a)
    # keys and values permuted together: the softmax sum over a segment does not depend on order
    np.testing.assert_allclose(oracle.attention(q, k[pk], v[pk], cu), base, rtol=0, atol=TOL)
    # query rows permuted: outputs follow their rows
    np.testing.assert_allclose(oracle.attention(q[pq], k, v, cu), base[pq], rtol=0, atol=TOL)


@_settings
@given(lengths=layouts, H=st.integers(1, 2), D=st.sampled_from([4, 8]), seed=st.integers(0, 2 ** 16))
def test_reordering_segments_moves_their_outputs(lengths, H, D, seed):
    q, k, v, cu = _inputs(lengths, H, D, seed)
    base = oracle.attention(q, k, v, cu)
    order = np.random.default_rng(seed + 2).permutation(len(lengths))
    rows = np.concatenate([np.arange(cu[i], cu[i + 1]) for i in order]).astype(np.int64)
    cu2 = np.concatenate([[0], np.cumsum([lengths[i] for i in order])]).astype(np.int32)
    np.testing.assert_allclose(oracle.attention(q[rows], k[rows], v[rows], cu2), base[rows], rtol=0, atol=TOL)


@_settings
@given(lengths=layouts, H=st.integers(2, 4), D=st.sampled_from([4, 8]), seed=st.integers(0, 2 ** 16))
def test_heads_are_independent(lengths, H, D, seed):
    q, k, v, cu = _inputs(lengths, H, D, seed)
    base = oracle.attention(q, k, v, cu)
    for h in range(H):
        one = oracle.attention(q[:, h:h + 1].copy(), k[:, h:h + 1].copy(), v[:, h:h + 1].copy(), cu)
        np.testing.assert_allclose(one[:, 0], base[:, h], rtol=0, atol=TOL)


@_settings
@given(lengths=layouts, D=st.sampled_from([4, 8, 16]), c=st.floats(0.25, 4.0), seed=st.integers(0, 2 ** 16))
def test_scale_folds_into_q_and_v_is_linear(lengths, D, c, seed):
    q, k, v, cu = _inputs(lengths, 2, D, seed)
    s = 1.0 / np.sqrt(D)
    base = oracle.attention(q, k, v, cu)
    np.testing.assert_allclose(oracle.attention(q * c, k, v, cu, scale=s / c), base, rtol=0, atol=1e-10)
    v2 = np.random.default_rng(seed + 3).standard_normal(v.shape)
    lin = oracle.attention(q, k, 2.0 * v - 3.0 * v2, cu)
    np.testing.assert_allclose(lin, 2.0 * base - 3.0 * oracle.attention(q, k, v2, cu), rtol=0, atol=1e-10)
