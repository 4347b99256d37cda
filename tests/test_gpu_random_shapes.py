"""Random small shapes, including V = 1 and V below one 16-byte vector, for
every entry point beside the fixed-length verify (which has its own 1000-call
case): each call against the oracle with the bar of its own test file."""

import numpy as np
import pytest
import torch

import oracle
from sampling_spec_verify_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"
VS = [1, 2, 7, 8, 9, 33, 1000, 2999]


@pytest.fixture(scope="module")
def ssv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sampling_spec_verify_gb300 as m
    m.lib()
    return m


def _case(rng, i):
    B = int(rng.integers(1, 6))
    K = int(rng.integers(0, 5))
    V = VS[i % len(VS)]
    dtype = torch.float32 if i % 2 else torch.bfloat16
    T = float(rng.choice([0.6, 1.0, 1.4]))
    w = synth.gaussian(B, K, V, sigma=2.0, noise=0.7, dtype=dtype, temperature=T, seed=1000 + i)
    return w, B, K, V, T


def test_overlap_and_diagnostics(ssv):
    rng = np.random.default_rng(71)
    for i in range(24):
        w, B, K, V, T = _case(rng, i)
        if K == 0:
            continue
        t, d = w.target.to(DEV), w.draft.to(DEV)
        o = ssv.overlap(t, d, T)
        dg = ssv.diagnostics(t, d, T)
        torch.cuda.synchronize()
        ro = oracle.overlap_stats(synth.f64(w.target[:, :K]), synth.f64(w.draft), T)
        rd = oracle.diagnostics(synth.f64(w.target[:, :K]), synth.f64(w.draft), T)
        np.testing.assert_allclose(o.alpha.cpu().numpy(), ro.alpha, rtol=1e-4, atol=1e-6, err_msg=str((B, K, V)))
        np.testing.assert_allclose(dg.entropy.cpu().numpy(), rd.entropy, rtol=1e-4, atol=1e-5)
        np.testing.assert_allclose(dg.kl.cpu().numpy(), rd.kl, rtol=1e-4, atol=1e-5)
        np.testing.assert_allclose(dg.alpha_target_only.cpu().numpy(), rd.alpha_to, rtol=1e-4, atol=1e-6)


def test_relaxed_ragged_and_tree(ssv):
    rng = np.random.default_rng(72)
    for i in range(24):
        w, B, K, V, T = _case(rng, i)
        t, d = w.target.to(DEV), w.draft.to(DEV)
        y, ua, uf = w.draft_tokens.to(DEV), w.u_accept.to(DEV), w.u_final.to(DEV)
        # relaxed
        kk, dl = int(rng.integers(0, 4)), float(rng.choice([0.5, 2.0, np.inf]))
        rx = ssv.verify_relaxed(t, d, y, uf, T, kk, dl)
        # ragged, lengths 0..K
        lengths = rng.integers(0, K + 1, size=B)
        off = np.zeros(B + 1, dtype=np.int32)
        off[1:] = np.cumsum(lengths + 1)
        tg = torch.cat([w.target[b, : l + 1] for b, l in enumerate(lengths)]).contiguous()
        nd = int(lengths.sum())
        dr = torch.cat([w.draft[b, :l] for b, l in enumerate(lengths)]).contiguous() if nd else None
        tk = torch.cat([w.draft_tokens[b, :l] for b, l in enumerate(lengths)]).contiguous()
        au = torch.cat([w.u_accept[b, :l] for b, l in enumerate(lengths)]).contiguous()
        rg = ssv.verify_ragged(tg.to(DEV), None if dr is None else dr.to(DEV), torch.from_numpy(off).to(DEV),
                               tk.to(DEV), au.to(DEV), uf, T)
        # a random tree over the K drafted tokens
        par = np.array([([-1] + [int(rng.integers(-1, j)) for j in range(1, K)])[:K] for _ in range(B)],
                       dtype=np.int32).reshape(B, K)
        tr = ssv.tree_verify_greedy(t, torch.from_numpy(par).to(DEV), y)
        torch.cuda.synchronize()
        rr = oracle.verify_relaxed(synth.f64(w.target), synth.f64(w.draft), w.draft_tokens.numpy(),
                                   w.u_final.numpy(), T, kk, dl)
        ok = ~rr.flagged
        tok = rx.tokens.cpu().numpy()
        assert (((tok == rr.tokens).all(axis=1)) | ~ok).all(), (i, B, K, V)
        for b, l in enumerate(lengths):
            ref = oracle.verify(synth.f64(w.target[b: b + 1, : l + 1]), synth.f64(w.draft[b: b + 1, :l]),
                                w.draft_tokens[b: b + 1, :l].numpy(), w.u_accept[b: b + 1, :l].numpy(),
                                w.u_final[b: b + 1].numpy(), T)
            if not ref.flagged[0]:
                assert rg.tokens[off[b]: off[b + 1]].cpu().tolist() == ref.tokens[0].tolist(), (i, b)
        rt = oracle.tree_verify_greedy(synth.f64(w.target), par, w.draft_tokens.numpy())
        assert tr.tokens.cpu().numpy().tolist() == rt.tokens.tolist(), (i, B, K, V)
        assert tr.n_accepted.cpu().numpy().tolist() == rt.n_accepted.tolist()


def test_truncation_small_vocabularies(ssv):
    rng = np.random.default_rng(73)
    for i in range(24):
        V = VS[i % len(VS)]
        dtype = torch.float32 if i % 2 else torch.bfloat16
        z = (torch.randn(3, V, generator=torch.Generator().manual_seed(i)) * 2).to(dtype)
        k = int(rng.integers(0, V + 2))
        p = float(rng.choice([0.3, 0.9, 1.0]))
        out = ssv.truncate_logits(z.to(DEV), 1.0, k, p)
        torch.cuda.synchronize()
        for r in range(3):
            want, near = oracle.truncate_logits(synth.f64(z[r]), 1.0, k, p)
            if near:
                continue
            got = np.isfinite(synth.f64(out[r].cpu()))
            assert (got == np.isfinite(want)).all(), (i, V, k, p, r)
