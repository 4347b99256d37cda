"""GPU parity of the diagnostics entry point (alpha, entropy, cross-entropy,
KL, target-only acceptance) against the fp64 oracle, through the C ABI.

Tolerances, from the kernel's fp32 arithmetic:
* every per-element exponent x = z s - c is rounded once (|x| < 64 in these
  workloads, so at most 2^-19 absolute) and 2^x is the hardware ex2 (a few
  ulp relative); alpha and p(argmax q) are sums or single terms of such
  values: 1e-4 relative plus 1e-6 absolute, as for the overlap;
* entropy and KL are sums of p x over up to 151936 tokens in fp32, with
  sum_v p |x| at most log2 V + |log2 q| weight, about 20 bits here; a
  rounding depth of about 30 additions gives under 2e-6 relative of that,
  so 1e-5 absolute plus 1e-4 relative;
* cross-entropy is entropy plus KL and takes the same bar.
The index y_hat = argmax q is taken on the stored logits on both sides
(scaling by 1/T > 0 keeps the order), so p(y_hat) has no tie ambiguity.
"""

import numpy as np
import pytest
import torch

import oracle
from sampling_spec_verify_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"
RTOL = 1e-4
ATOL_P = 1e-6    # alpha, p(y_hat)
ATOL_LOG = 1e-5  # entropy, cross-entropy, KL


@pytest.fixture(scope="module")
def ssv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sampling_spec_verify_gb300 as m
    m.lib()
    return m


def _compare(d, ref, rows=None):
    got = {
        "alpha": d.alpha, "entropy": d.entropy, "cross_entropy": d.cross_entropy, "kl": d.kl,
        "alpha_to": d.alpha_target_only,
    }
    for name, t in got.items():
        g = t.cpu().numpy().astype(np.float64)
        if rows is not None:
            g = g[rows]
        want = getattr(ref, name)
        atol = ATOL_LOG if name in ("entropy", "cross_entropy", "kl") else ATOL_P
        np.testing.assert_allclose(g, want, rtol=RTOL, atol=atol, err_msg=name)


@pytest.mark.parametrize("B,K,V,dtype,T", [
    (3, 4, 3000, torch.float32, 1.0),
    (4, 5, 20011, torch.bfloat16, 0.8),   # ragged slice tail, element-wise staging
    (2, 3, 999, torch.float32, 0.6),
    (2, 2, 50000, torch.bfloat16, 1.7),
])
def test_small_against_oracle(ssv, B, K, V, dtype, T):
    w = synth.gaussian(B, K, V, sigma=2.0, noise=0.5, dtype=dtype, temperature=T, seed=11 * B + K + V,
                       bonus=False, draft_tokens=False)
    d = ssv.diagnostics(w.target.to(DEV), w.draft.to(DEV), w.temperature)
    torch.cuda.synchronize()
    assert int(d.status.item()) == 0
    ref = oracle.diagnostics(synth.f64(w.target), synth.f64(w.draft), w.temperature)
    _compare(d, ref)


def test_entropy_mix_full_size_verify_layout(ssv):
    """The verify batch (B=32, K=4, V=151936, per-row sigma in {1, 2, 4})
    read through its [B, K+1, V] target tensor."""
    w = synth.entropy_mix(seed=4242)
    B, K, V = w.shape
    d = ssv.diagnostics(w.target.to(DEV), w.draft.to(DEV), 1.0)
    torch.cuda.synchronize()
    assert int(d.status.item()) == 0
    ref = oracle.diagnostics(synth.f64(w.target[:, :K]), synth.f64(w.draft), 1.0)
    _compare(d, ref)
    # higher target entropy, lower target-only acceptance (the pages' claim),
    # visible across the three sigma groups
    h = d.entropy.cpu().numpy().mean(axis=1)
    ato = d.alpha_target_only.cpu().numpy().mean(axis=1)
    assert np.corrcoef(h, ato)[0, 1] < 0


def test_e2e_batch_full_size_sampled_rows(ssv):
    w = synth.e2e(seed=4343)
    B, K, V = w.shape
    d = ssv.diagnostics(w.target.to(DEV), w.draft.to(DEV), 1.0)
    torch.cuda.synchronize()
    assert int(d.status.item()) == 0
    rows = [0, 77, 131, 255]
    ref = oracle.diagnostics(synth.f64(w.target), synth.f64(w.draft), 1.0, rows=rows)
    _compare(d, ref, rows=rows)
    # properties at every row: CE = H + KL, KL >= 0, Pinsker, alpha_TO <= max p
    H, CE, KL = (t.cpu().numpy().astype(np.float64) for t in (d.entropy, d.cross_entropy, d.kl))
    a = d.alpha.cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(CE, H + KL, rtol=1e-6, atol=1e-6)
    assert (KL > -1e-6).all()
    assert ((1.0 - a) <= np.sqrt(0.5 * np.maximum(KL, 0.0)) + 1e-5).all()


def test_identical_rows_and_argmax_ties(ssv):
    """q = p: alpha 1, KL 0, CE = H, alpha_TO = max p.  Drafts with a repeated
    maximum pick the smallest index."""
    B, K, V = 2, 3, 4099
    g = torch.Generator().manual_seed(5)
    t = torch.randn(B, K, V, generator=g).to(torch.bfloat16)
    dr = t.clone()
    dr[0, 1, 17] = 9.0
    dr[0, 1, 4000] = 9.0   # tie: y_hat = 17
    dr[1, 2, 3] = 7.5
    dr[1, 2, 2] = 7.5      # tie: y_hat = 2
    d = ssv.diagnostics(t.to(DEV), dr.to(DEV), 1.0)
    torch.cuda.synchronize()
    ref = oracle.diagnostics(synth.f64(t), synth.f64(dr), 1.0)
    _compare(d, ref)
    same = [(0, 0), (0, 2), (1, 0), (1, 1)]
    for b, k in same:
        assert abs(float(d.alpha[b, k]) - 1.0) <= 2e-6
        assert abs(float(d.kl[b, k])) <= 1e-6
    p01 = oracle.softmax_t(synth.f64(t)[0, 1], 1.0)
    assert abs(float(d.alpha_target_only[0, 1]) - p01[17]) <= 1e-6 + 1e-4 * p01[17]


def test_masked_tokens(ssv):
    """-inf logits: p = 0 tokens add nothing to H or KL; a token with q = 0 < p
    makes KL and CE infinite."""
    B, K, V = 1, 3, 5003
    g = torch.Generator().manual_seed(6)
    t = torch.randn(B, K, V, generator=g)
    dr = t + 0.3 * torch.randn(B, K, V, generator=g)
    t[0, 0, :2000] = -float("inf")          # target masked, draft not: finite
    t[0, 1, 100:300] = -float("inf")
    dr[0, 1, 100:300] = -float("inf")       # both masked: finite
    dr[0, 2, 42] = -float("inf")            # q = 0 < p: infinite KL and CE
    d = ssv.diagnostics(t.to(DEV), dr.to(DEV), 1.0)
    torch.cuda.synchronize()
    assert int(d.status.item()) == 0
    ref = oracle.diagnostics(synth.f64(t), synth.f64(dr), 1.0)
    assert np.isinf(ref.kl[0, 2]) and np.isinf(ref.cross_entropy[0, 2])
    assert np.isposinf(d.kl.cpu().numpy()[0, 2]) and np.isposinf(d.cross_entropy.cpu().numpy()[0, 2])
    for name in ("alpha", "entropy", "alpha_target_only"):
        got = getattr(d, name).cpu().numpy()
        want = getattr(ref, "alpha_to" if name == "alpha_target_only" else name)
        atol = ATOL_LOG if name == "entropy" else ATOL_P
        np.testing.assert_allclose(got, want, rtol=RTOL, atol=atol, err_msg=name)
    for name in ("kl", "cross_entropy"):
        np.testing.assert_allclose(getattr(d, name).cpu().numpy()[0, :2], getattr(ref, name)[0, :2],
                                   rtol=RTOL, atol=ATOL_LOG, err_msg=name)


def test_bad_rows_nan_and_status(ssv):
    B, K, V = 2, 2, 1024
    g = torch.Generator().manual_seed(7)
    t = torch.randn(B, K, V, generator=g)
    dr = torch.randn(B, K, V, generator=g)
    t[1, 0, 5] = float("nan")
    d = ssv.diagnostics(t.to(DEV), dr.to(DEV), 1.0)
    torch.cuda.synchronize()
    assert int(d.status.item()) & ssv.DEV_BAD_LOGITS
    for f in (d.alpha, d.entropy, d.cross_entropy, d.kl, d.alpha_target_only):
        a = f.cpu().numpy()
        assert np.isnan(a[1, 0])
        assert np.isfinite(a[0]).all() and np.isfinite(a[1, 1])
    ref = oracle.diagnostics(synth.f64(t), synth.f64(dr), 1.0, rows=[0])
    np.testing.assert_allclose(d.entropy.cpu().numpy()[:1], ref.entropy, rtol=RTOL, atol=ATOL_LOG)


def test_optional_outputs_and_workspace_reuse(ssv):
    """Outputs passed as None are not written; a workspace left zero by one
    call serves the next and gives the same bits."""
    B, K, V = 3, 4, 8000
    w = synth.gaussian(B, K, V, sigma=2.0, noise=0.5, dtype=torch.bfloat16, temperature=1.0, seed=99,
                       bonus=False, draft_tokens=False)
    t, dr = w.target.to(DEV), w.draft.to(DEV)
    ws = torch.zeros(ssv.lib().spec_diagnostics_workspace_bytes(B, K, V), dtype=torch.uint8, device=DEV)
    full = ssv.diagnostics(t, dr, 1.0, workspace=ws)
    e = lambda: torch.full((B, K), -7.0, device=DEV)  # noqa: E731
    part = ssv.DiagOutput(None, e(), None, None, e(), torch.zeros(1, dtype=torch.int32, device=DEV))
    ssv.diagnostics(t, dr, 1.0, out=part, workspace=ws)
    again = ssv.diagnostics(t, dr, 1.0, workspace=ws)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero()) == 0
    assert torch.equal(part.entropy, full.entropy)
    assert torch.equal(part.alpha_target_only, full.alpha_target_only)
    for f in ("alpha", "entropy", "cross_entropy", "kl", "alpha_target_only"):
        assert torch.equal(getattr(again, f), getattr(full, f)), f


def test_empty_and_invalid(ssv):
    t = torch.zeros(0, 2, 16, device=DEV)
    d = ssv.diagnostics(t, t, 1.0)
    assert d.alpha.numel() == 0
    x = torch.randn(1, 2, 16, device=DEV)
    with pytest.raises(ssv.SpecError):
        ssv.diagnostics(x, x, 0.0)
