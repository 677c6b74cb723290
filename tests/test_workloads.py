"""The synthetic input recipe (CPU only): the five workloads have the shapes,
sizes, group layouts and value distributions stated for them, and their
generators are seeded and reproducible."""

import math

import numpy as np
import pytest
import torch

import workloads


def test_sizes_and_layouts():
    sizes = {1: 262_144, 2: 213_909_504, 3: 520_093_696, 4: 872_415_232, 5: 872_415_232}
    for k, n in sizes.items():
        assert workloads.get(k).numel == n, k
    w2 = workloads.get(2)
    assert len(w2.matrices) == 24 and w2.groups == 24 and not w2.ns
    assert [m.name.split(".")[1] for m in w2.matrices[-3:]] == ["q", "k", "v"]   # cut inside the 4th layer
    w3 = workloads.get(3)
    assert w3.groups == 11 and w3.q8_kind == "int8"
    qkv = w3.matrices[0]
    third = qkv.numel // 3
    assert [(s.start, s.length, s.group_id) for s in w3.segments[:3]] == [(0, third, 0), (third, third, 1),
                                                                         (2 * third, third, 2)]
    w4 = workloads.get(4)
    assert (w4.P, w4.tile, w4.steps, len(w4.matrices)) == (5, (1, 8), 20, 28)
    assert w4.eta_full == 0.02 and abs(w4.eta_block - 0.02 / math.sqrt(8)) < 1e-15
    # every 1 x 8 column tile of every matrix is whole 256-element runs
    assert all(m.cols % 8 == 0 and (m.cols // 8) % 256 == 0 for m in w4.matrices)
    assert workloads.get(5).carrier and all(m.cols % 32 == 0 for m in workloads.get(5).matrices)


def _grad(k, step=1, rows=1024, cols=512, index=0):
    w = workloads.get(k)
    return workloads.make_grad(w, index, step, matrix=workloads.Matrix("s", rows, cols)).float().numpy()


def test_gradient_distributions():
    # c1: N(0, 1e-3^2)
    g = _grad(1)
    assert abs(g.std() - 1e-3) < 2e-5 and abs(g.mean()) < 1e-5
    # c2 / c4: z * exp(N(0, 1)) per row -- the log of each row's spread is N(0, 1)
    for k in (2, 4):
        ls = np.log(_grad(k).std(axis=1))
        assert abs(ls.mean()) < 0.1 and abs(ls.std() - 1.0) < 0.08, k
    # c5: z * exp(1.5 N(0, 1)) per column
    ls = np.log(_grad(5, rows=512, cols=1024).std(axis=0))
    assert abs(ls.mean()) < 0.15 and abs(ls.std() - 1.5) < 0.1
    # c3: N(0, 1) with about 0.1% of the entries scaled by 100
    g = _grad(3, rows=2048, cols=1024)
    big = np.abs(g) > 8.0
    assert 0.0006 < big.mean() < 0.0014
    assert abs(g[~big].std() - 1.0) < 0.01


def test_generators_are_seeded_and_distinct():
    a, b = _grad(4, step=3), _grad(4, step=3)
    assert np.array_equal(a, b)                                    # reproducible
    assert not np.array_equal(a, _grad(4, step=4))                 # per step
    assert not np.array_equal(a, _grad(4, step=3, index=1))        # per matrix
    assert workloads.grad_seed(4, 7) == 4007
    w = workloads.get(4)
    wt = workloads.make_weight(w, 1)
    assert torch.equal(wt, workloads.make_weight(w, 1))
    assert abs(float(wt.std()) - 0.02) < 2e-4


@pytest.mark.parametrize("q8_kind", ["int8", "uint8"])
def test_states(q8_kind):
    m = workloads.Matrix("t", 300, 100)
    q, a = workloads.zero_state(m, q8_kind)
    assert q.numel() == 30000 and a.numel() == 118 and float(a.abs().max()) == 0.0
    assert int(q[0]) == (0 if q8_kind == "int8" else 128)
    q, a = workloads.random_state(m, 5, q8_kind)
    vals = q.to(torch.int32) - (0 if q8_kind == "int8" else 128)
    assert int(vals.min()) >= -127 and int(vals.max()) <= 127
    la = torch.log(a)
    assert float(la.min()) >= -9.0 and float(la.max()) <= 3.0


def test_code_kind_variant():
    # the grouped workload names both code kinds: the uint8 variant differs
    # from the default only in its state encoding
    a, b = workloads.get(3), workloads.get(3, q8_kind="uint8")
    assert a.q8_kind == "int8" and b.q8_kind == "uint8"
    assert a.matrices == b.matrices and a.segments == b.segments and a.ns_slices == b.ns_slices
    with pytest.raises(ValueError):
        workloads.get(3, q8_kind="int4")
