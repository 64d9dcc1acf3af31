"""The seeded input generators: shapes, determinism and the routing structure
each workload asks for (no GPU, no oracle)."""
import numpy as np

from unpermute_routing_indices_gb300 import workloads as wl


def test_tiny_routing_is_distinct_topk_with_softmax():
    idx, probs, E = wl.routing("tiny")
    assert idx.shape == (16, 4) and E == 32
    assert all(len(set(r)) == 4 for r in idx.tolist())
    np.testing.assert_allclose(probs.sum(1), 1.0, rtol=1e-6)
    assert np.all(np.diff(probs, axis=1) <= 0)           # larger logit first


def test_generators_are_deterministic():
    a = wl.routed("tiny")
    b = wl.routed("tiny")
    for k in ("idx", "probs", "x", "g_y", "g_out_probs"):
        np.testing.assert_array_equal(a[k], b[k])
    assert a["x"].dtype == np.uint16 and a["x"].shape == (16, 64)


def test_skewed_routing_has_hot_and_empty_experts():
    idx, _, E = wl.routing("skewed", T=2048)
    counts = np.bincount(idx.ravel(), minlength=E)
    assert (counts == 0).sum() >= 1
    assert counts.max() > 8 * counts.sum() / E


def test_group_limited_routing_uses_at_most_four_groups():
    idx, probs, E = wl.routing("large", T=512)
    groups = idx // (E // 8)
    assert max(len(set(r)) for r in groups.tolist()) <= 4
    assert all(len(set(r)) == 8 for r in idx.tolist())
    np.testing.assert_allclose(probs.sum(1), 1.0, rtol=1e-6)


def test_chunk_layout():
    for N in (8192, 32768):
        sizes, order = wl.chunk_layout(N)
        assert sizes.shape == (128,) and sizes.sum() == N
        assert (sizes == 0).sum() >= 16
        assert sorted(order.tolist()) == list(range(128))
        assert order[0 * 8 + 1] == 1 * 16 + 0              # expert 0, rank 1
