"""GPU parity of the relaxed (LOSSY) verify against the fp64 oracle.

Bar: tokens and accepted counts bit-exact on rows the oracle does not flag
(gap within 1e-6 of -delta, or a CDF boundary within 1e-6); alpha within
1e-4 relative + 1e-6.
"""

import numpy as np
import pytest
import torch

import oracle
from sampling_spec_verify_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"
INF = float("inf")


@pytest.fixture(scope="module")
def ssv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sampling_spec_verify_gb300 as m
    m.lib()
    return m


def _check(out, ref, rows=None):
    tok = out.tokens.cpu().numpy()
    n = out.n_accepted.cpu().numpy()
    if rows is not None:
        tok, n = tok[rows], n[rows]
    ok = ~ref.flagged
    bad = np.nonzero(ok & ((tok != ref.tokens).any(axis=1) | (n != ref.n_accepted)))[0]
    assert bad.size == 0, f"rows {bad[:8]}: gpu {tok[bad[:2]]} {n[bad[:2]]} vs {ref.tokens[bad[:2]]} {ref.n_accepted[bad[:2]]}"
    a = out.alpha.cpu().numpy()
    if rows is not None:
        a = a[rows]
    np.testing.assert_allclose(a, ref.alpha, rtol=1e-4, atol=1e-6)
    return int(ref.flagged.sum())


@pytest.mark.parametrize("B,K,V,dtype,T,k,delta", [
    (16, 4, 3000, torch.float32, 1.0, 5, INF),
    (16, 4, 3000, torch.float32, 1.0, 0, 1.5),
    (12, 5, 20011, torch.bfloat16, 0.8, 20, 2.0),   # unaligned rows
    (8, 3, 999, torch.float32, 0.7, 1, INF),        # top-1: the greedy acceptance
    (8, 3, 4096, torch.bfloat16, 1.0, 0, INF),      # no condition: all accepted
])
def test_against_oracle(ssv, B, K, V, dtype, T, k, delta):
    w = synth.gaussian(B, K, V, sigma=2.0, noise=0.8, dtype=dtype, temperature=T, seed=B * 7 + K + k)
    t, d, y, _, uf = (w.target.to(DEV), w.draft.to(DEV), w.draft_tokens.to(DEV), None, w.u_final.to(DEV))
    out = ssv.verify_relaxed(t, d, y, uf, T, k, delta)
    torch.cuda.synchronize()
    assert int(out.status.item()) == 0
    ref = oracle.verify_relaxed(synth.f64(w.target), synth.f64(w.draft), w.draft_tokens.numpy(),
                                w.u_final.numpy(), T, k, delta)
    _check(out, ref)
    if k == 0 and delta == INF:
        assert (out.n_accepted.cpu().numpy() == K).all()


def test_full_size_verify_batch(ssv):
    w = synth.entropy_mix(seed=717)
    out = ssv.verify_relaxed(w.target.to(DEV), w.draft.to(DEV), w.draft_tokens.to(DEV), w.u_final.to(DEV),
                             1.0, 8, 3.0)
    torch.cuda.synchronize()
    ref = oracle.verify_relaxed(synth.f64(w.target), synth.f64(w.draft), w.draft_tokens.numpy(),
                                w.u_final.numpy(), 1.0, 8, 3.0)
    _check(out, ref)
    # the relaxed rule accepts at least as often as ... itself with a tighter top-k
    tight = ssv.verify_relaxed(w.target.to(DEV), w.draft.to(DEV), w.draft_tokens.to(DEV), w.u_final.to(DEV),
                               1.0, 2, 3.0)
    torch.cuda.synchronize()
    assert (out.n_accepted >= tight.n_accepted).all()


def test_ties_rank_by_index_and_bad_token(ssv):
    B, K, V = 2, 2, 1024
    t = torch.full((B, K + 1, V), -2.0)
    t[:, :, 10] = 3.0
    t[:, :, 20] = 3.0   # tie with 10: 20 ranks second
    d = t[:, :K].clone()
    y = torch.tensor([[20, 10], [10, V + 3]], dtype=torch.int32)
    uf = torch.tensor([0.3, 0.6])
    out = ssv.verify_relaxed(t.to(DEV), d.to(DEV), y.to(DEV), uf.to(DEV), 1.0, 1, INF)
    torch.cuda.synchronize()
    ref = oracle.verify_relaxed(synth.f64(t), synth.f64(d), y.numpy(), uf.numpy(), 1.0, 1, INF)
    assert out.n_accepted.cpu().tolist() == ref.n_accepted.tolist() == [0, 1]
    assert int(out.status.item()) & ssv.DEV_BAD_TOKEN
    assert out.tokens.cpu().numpy().tolist() == ref.tokens.tolist()


def test_invalid(ssv):
    w = synth.gaussian(2, 2, 64, dtype=torch.float32, temperature=1.0, seed=1)
    args = (w.target.to(DEV), w.draft.to(DEV), w.draft_tokens.to(DEV), w.u_final.to(DEV))
    with pytest.raises(ssv.SpecError):
        ssv.verify_relaxed(*args, 0.0, 2, 1.0)   # T > 0 only
    with pytest.raises(ssv.SpecError):
        ssv.verify_relaxed(*args, 1.0, 2, -1.0)  # delta >= 0
