"""The two-pass sweep (pass A from HBM, pass C from L2) against the oracle and
against the single-read sweep, over cluster sizes, chunked slices, ring
depths and every mode it serves: sampling verify with and without the
overlap, greedy verify, overlap statistics and the E2E-TV forward pass.

Bars as in test_gpu_parity: tokens and counts bit-exact on every row the
oracle does not flag; floats within 1e-4 relative plus 1e-6 absolute."""

import numpy as np
import pytest
import torch

import oracle
from sampling_spec_verify_gb300 import synth

pytestmark = pytest.mark.gpu

RTOL, ATOL = 1e-4, 1e-6
DEV = "cuda"


@pytest.fixture(scope="module")
def ssv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sampling_spec_verify_gb300 as m
    m.lib()
    yield m
    m.set_kernel_override(0)
    m.set_launch_override(0, 0)


def _dev(w):
    return (w.target.to(DEV), w.draft.to(DEV), w.draft_tokens.to(DEV), w.u_accept.to(DEV), w.u_final.to(DEV))


def _oracle(w, with_draft=True):
    return oracle.verify(synth.f64(w.target), synth.f64(w.draft) if with_draft else None,
                         w.draft_tokens.numpy(), w.u_accept.numpy(), w.u_final.numpy(), w.temperature)


def _check(out, ref, check_alpha=True):
    tok, n = out.tokens.cpu().numpy(), out.n_accepted.cpu().numpy()
    ok = ~ref.flagged
    bad = np.nonzero(ok & ((tok != ref.tokens).any(axis=1) | (n != ref.n_accepted)))[0]
    assert bad.size == 0, f"rows {bad[:8]}: gpu {tok[bad[:2]]} vs oracle {ref.tokens[bad[:2]]}"
    if check_alpha and out.alpha is not None:
        np.testing.assert_allclose(out.alpha.cpu().numpy(), ref.alpha, rtol=RTOL, atol=ATOL)


def _run(ssv, kernel, S, nst, fn):
    ssv.set_kernel_override(kernel)
    ssv.set_launch_override(S, nst)
    try:
        out = fn()
        torch.cuda.synchronize()
    finally:
        ssv.set_kernel_override(0)
        ssv.set_launch_override(0, 0)
    return out


# B, K, V, dtype, T, S (0 = automatic), stages cap (0 = automatic)
SHAPES = [
    (4, 3, 151936, torch.bfloat16, 1.0, 1, 0),    # one CTA per row: 10 chunks per slice
    (6, 4, 151936, torch.bfloat16, 0.7, 2, 0),    # CTA pairs: 5 chunks each
    (5, 7, 129280, torch.bfloat16, 1.0, 3, 2),    # uneven slices of 3 chunks, a two-stage ring
    (9, 2, 40000, torch.bfloat16, 1.0, 16, 0),    # 16 CTAs, short slices
    (3, 5, 24000, torch.float32, 1.3, 1, 1),      # fp32, 3 chunks through a one-stage ring
    (2, 4, 8, torch.bfloat16, 1.0, 16, 0),        # V below one vector per CTA: empty slices
    (3, 0, 5000, torch.bfloat16, 1.0, 0, 0),      # K = 0: the bonus draw only
    (2, 33, 1024, torch.float32, 0.9, 0, 0),      # K + 1 above one warp
    (64, 4, 30000, torch.bfloat16, 1.0, 2, 0),    # more rows than clusters: row groups
]


@pytest.mark.parametrize("B,K,V,dtype,T,S,nst", SHAPES)
def test_two_pass_against_oracle_and_single_read(ssv, B, K, V, dtype, T, S, nst):
    w = synth.gaussian(B, K, V, sigma=2.0, noise=0.6, dtype=dtype, temperature=T, seed=B * 97 + K * 13 + V)
    args = _dev(w)
    two = _run(ssv, 2, S, nst, lambda: ssv.verify(*args, w.temperature))
    one = _run(ssv, 1, 0, 0, lambda: ssv.verify(*args, w.temperature))
    ref = _oracle(w)
    _check(two, ref)
    _check(one, ref)
    assert int(two.status.item()) == 0
    if K:
        np.testing.assert_allclose(two.alpha.cpu().numpy(), one.alpha.cpu().numpy(), rtol=RTOL, atol=ATOL)
    # the two-pass launch shape reported for the forced cluster size
    if S:
        ssv.set_kernel_override(2)
        ssv.set_launch_override(S, nst)
        try:
            assert ssv.launch_shape(dtype, B * (K + 1), V)[0] == S
        finally:
            ssv.set_launch_override(0, 0)
            ssv.set_kernel_override(0)


@pytest.mark.parametrize("S", [1, 2, 5, 16])
def test_two_pass_greedy(ssv, S):
    B, K, V = 5, 4, 60000
    w = synth.gaussian(B, K, V, sigma=2.0, noise=0.3, dtype=torch.bfloat16, temperature=0.0, seed=300 + S)
    t, d, y = w.target.to(DEV), w.draft.to(DEV), w.draft_tokens.to(DEV)
    # ties across slices and chunks: the smallest index wins
    t[0, 0, 100] = 30.0
    t[0, 0, 59000] = 30.0
    t[1, 1, 4000] = 30.0
    t[1, 1, 3999] = 30.0
    with_a = _run(ssv, 2, S, 0, lambda: ssv.verify(t, d, y, None, None, 0.0))
    no_a = _run(ssv, 2, S, 0, lambda: ssv.verify(t, None, y, None, None, 0.0))
    ref = oracle.verify(t.double().cpu().numpy(), d.double().cpu().numpy(), w.draft_tokens.numpy(),
                        np.zeros((B, K)), np.zeros(B), 0.0)
    for out in (with_a, no_a):
        assert (out.tokens.cpu().numpy() == ref.tokens).all()
        assert (out.n_accepted.cpu().numpy() == ref.n_accepted).all()
        assert int(out.status.item()) == 0
    np.testing.assert_array_equal(with_a.alpha.cpu().numpy(), ref.alpha)
    assert int(with_a.tokens[0, 0]) == 100 or int(with_a.n_accepted[0]) > 0


@pytest.mark.parametrize("S", [0, 1, 3])
def test_two_pass_overlap_and_e2e(ssv, S):
    B, K, V = 6, 5, 70000
    w = synth.gaussian(B, K, V, sigma=2.0, noise=0.5, dtype=torch.bfloat16, temperature=1.0, seed=500 + S,
                       bonus=False, draft_tokens=False)
    t, d = w.target.to(DEV), w.draft.to(DEV)
    o = _run(ssv, 2, S, 0, lambda: ssv.overlap(t, d, 1.0))
    e = _run(ssv, 2, S, 0, lambda: ssv.e2e_tv_fwd_bwd(t, d, 1.0, grad_scale=-1.0))
    ro = oracle.overlap_stats(synth.f64(w.target), synth.f64(w.draft), 1.0)
    for got, want in ((o.alpha, ro.alpha), (o.tv, ro.tv), (o.prefix_survival, ro.prefix_survival),
                      (o.expected_accepted, ro.expected_accepted), (e.alpha, ro.alpha)):
        np.testing.assert_allclose(got.cpu().numpy(), want, rtol=RTOL, atol=ATOL)
    L, _ = oracle.e2e_tv_loss(synth.f64(w.target), synth.f64(w.draft), 1.0)
    assert abs(float(e.loss.item()) - L) <= ATOL + RTOL * abs(L)
    rg, amb = oracle.e2e_tv_grad(synth.f64(w.target), synth.f64(w.draft), 1.0, grad_scale=-1.0)
    g = e.grad.cpu().numpy()
    bad = (np.abs(g - rg) > ATOL + RTOL * np.abs(rg)) & ~amb
    assert not bad.any(), f"{bad.sum()} gradient elements off"


def test_two_pass_without_alpha_and_deterministic(ssv):
    B, K, V = 40, 5, 50000
    w = synth.gaussian(B, K, V, sigma=1.5, noise=0.9, dtype=torch.bfloat16, temperature=1.0, seed=77)
    args = _dev(w)
    L = ssv.lib()
    ws = torch.zeros(L.spec_verify_workspace_bytes(B, K, V), dtype=torch.uint8, device=DEV)
    a = _run(ssv, 2, 2, 0, lambda: ssv.verify(*args, 1.0, workspace=ws))
    b = _run(ssv, 2, 2, 0, lambda: ssv.verify(*args, 1.0, workspace=ws))
    c = _run(ssv, 2, 2, 0, lambda: ssv.verify(*args, 1.0, want_alpha=False, workspace=ws))
    assert torch.equal(a.tokens, b.tokens) and torch.equal(a.alpha, b.alpha)
    assert torch.equal(a.tokens, c.tokens) and torch.equal(a.n_accepted, c.n_accepted)
    assert c.alpha is None
    assert int(ws.count_nonzero().item()) == 0
    _check(a, _oracle(w))


def test_two_pass_rejections_everywhere(ssv):
    """Disjoint draft mass: every position rejects, so every row draws its
    correction at position 0 and later positions skip or draw unused."""
    B, K, V = 20, 4, 20000
    w = synth.gaussian(B, K, V, sigma=3.0, noise=6.0, dtype=torch.bfloat16, temperature=1.0, seed=91)
    args = _dev(w)
    out = _run(ssv, 2, 0, 0, lambda: ssv.verify(*args, 1.0))
    ref = _oracle(w)
    _check(out, ref)
    assert (ref.n_accepted < K).sum() >= B // 2


def test_kernel_choice_by_bytes_read(ssv):
    """The automatic choice: the two-pass sweep (608 threads) for calls that
    read at least 200 MB of logits, the single-read sweep (256) below."""
    assert ssv.launch_shape(torch.bfloat16, 128 * 8, 129280)[1] == 608   # 1024 units x 2 rows: 530 MB
    assert ssv.launch_shape(torch.bfloat16, 32 * 5, 151936)[1] == 256    # 97 MB
    ssv.set_kernel_override(2)
    try:
        assert ssv.launch_shape(torch.bfloat16, 32 * 5, 151936)[1] == 608
    finally:
        ssv.set_kernel_override(0)
