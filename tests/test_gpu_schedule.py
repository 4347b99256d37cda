"""GPU parity of verify-length scheduling against the fp64 oracle.

Bar: lengths bit-exact wherever the oracle reports no near tie between two
total lengths (throughputs within 1e-9 relative); Theta and tau within
1e-6 relative (they are returned as float32).
"""

import numpy as np
import pytest
import torch

import oracle
from sampling_spec_verify_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def ssv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sampling_spec_verify_gb300 as m
    m.lib()
    return m


def _survivals(rng, R, L):
    return np.cumprod(rng.uniform(0.3, 1.0, size=(R, L)), axis=1).astype(np.float32)


def _sps(rng, n):
    # decode steps per second falling with the batch, with cliffs (graph buckets)
    b = np.arange(n, dtype=np.float64)
    s = 2000.0 / (1.0 + b / rng.uniform(64.0, 512.0))
    for c in rng.choice(np.arange(1, n), size=min(6, n - 1), replace=False):
        s[c:] *= rng.uniform(0.8, 0.97)
    return s.astype(np.float32)


def _run(ssv, a, sps):
    lengths, obj = ssv.schedule_lengths(torch.from_numpy(a).to(DEV), torch.from_numpy(sps).to(DEV))
    torch.cuda.synchronize()
    return lengths.cpu().numpy(), obj.cpu().numpy()


def _check(ssv, a, sps):
    ref = oracle.schedule_lengths(a.astype(np.float64), sps.astype(np.float64))
    got, obj = _run(ssv, a, sps)
    if not ref.near:
        np.testing.assert_array_equal(got, ref.lengths)
    assert obj[0] == pytest.approx(ref.theta, rel=1e-6)
    assert obj[1] == pytest.approx(ref.tau, rel=1e-6)
    assert ((got >= 0) & (got <= a.shape[1])).all()
    return ref


@pytest.mark.parametrize("R,L", [(1, 1), (3, 2), (7, 4), (64, 7), (256, 4), (1000, 16), (1024, 16), (16384, 1)])
def test_random_against_oracle(ssv, R, L):
    rng = np.random.default_rng(R * 100 + L)
    a = _survivals(rng, R, L)
    sps = _sps(rng, R * (1 + L) + 1)
    _check(ssv, a, sps)


def test_hand_example(ssv):
    got, obj = _run(ssv, np.array([[0.9, 0.5], [0.6, 0.1]], np.float32),
                    np.array([0, 0, 100, 95, 80, 78, 60], np.float32))
    assert got.tolist() == [2, 1]
    assert obj[0] == pytest.approx(312.0) and obj[1] == pytest.approx(4.0)


def test_ties_and_flat_and_cliff(ssv):
    a = np.full((6, 3), 0.5, np.float32)  # all equal: taken in (row, position) order
    sps = np.full(6 * 4 + 1, 10.0, np.float32)
    sps[6 + 7 + 1:] = 0.0                 # B <= 13: room for 7 drafted tokens only
    got, _ = _run(ssv, a, sps)
    ref = oracle.schedule_lengths(a, sps)
    assert got.tolist() == ref.lengths.tolist() == [3, 3, 1, 0, 0, 0]
    flat = np.full(6 * 4 + 1, 3.0, np.float32)
    got, _ = _run(ssv, a, flat)
    assert got.tolist() == [3] * 6


def test_from_overlap_prefix_survival(ssv):
    """The scheduler fed by the overlap kernel's prefix survivals of the
    verify batch (B=32, K=4, V=151936)."""
    w = synth.entropy_mix(seed=31)
    B, K, V = w.shape
    o = ssv.overlap(w.target.to(DEV), w.draft.to(DEV), 1.0)
    torch.cuda.synchronize()
    a = o.prefix_survival.cpu().numpy()
    rng = np.random.default_rng(5)
    sps = _sps(rng, B * (1 + K) + 1)
    lengths, obj = ssv.schedule_lengths(o.prefix_survival, torch.from_numpy(sps).to(DEV))
    torch.cuda.synchronize()
    ref = oracle.schedule_lengths(a.astype(np.float64), sps.astype(np.float64))
    if not ref.near:
        np.testing.assert_array_equal(lengths.cpu().numpy(), ref.lengths)
    assert float(obj[0]) == pytest.approx(ref.theta, rel=1e-6)


def test_nan_and_invalid(ssv):
    a = np.array([[0.9, np.nan], [0.5, 0.4]], np.float32)
    sps = np.array([0, 0, 10, 9.5, 9.2, 9.0, 8.0], np.float32)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    lengths, _ = ssv.schedule_lengths(torch.from_numpy(a).to(DEV), torch.from_numpy(sps).to(DEV), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & ssv.DEV_BAD_LOGITS
    ref = oracle.schedule_lengths(np.nan_to_num(a, nan=0.0), sps)
    assert lengths.cpu().tolist() == ref.lengths.tolist()
    with pytest.raises(ssv.SpecError):  # table too short
        ssv.schedule_lengths(torch.from_numpy(a).to(DEV), torch.from_numpy(sps[:5]).to(DEV))
    with pytest.raises(ssv.SpecError):  # beyond the shared-memory limit
        ssv.schedule_lengths(torch.zeros((16385, 1), device=DEV), torch.zeros(40000, device=DEV))
