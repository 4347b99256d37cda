"""GPU parity: the CUDA path, called through the C ABI, against the fp64
oracle on the same seeded inputs.

Bars (written out here):
* integer outputs (tokens, accepted counts) bit-exact on every row the oracle
  does not flag (|u - p/q| or a residual-CDF boundary within 1e-6);
* floats (alpha, TV, survival, loss, gradient) within 1e-4 relative plus
  1e-6 absolute of the fp64 value;
* the gradient is compared element by element except where the oracle marks
  the indicator 1[q < p] as within 1e-6 of flipping.
"""

import numpy as np
import pytest
import torch

import oracle
from sampling_spec_verify_gb300 import synth

pytestmark = pytest.mark.gpu

RTOL, ATOL = 1e-4, 1e-6


@pytest.fixture(scope="module")
def ssv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sampling_spec_verify_gb300 as m
    m.lib()
    return m


DEV = "cuda"


def to_dev(w):
    return (w.target.to(DEV), w.draft.to(DEV), w.draft_tokens.to(DEV), w.u_accept.to(DEV), w.u_final.to(DEV))


def oracle_verify(w, T=None, rows=None, with_draft=True):
    T = w.temperature if T is None else T
    return oracle.verify(synth.f64(w.target), synth.f64(w.draft) if with_draft else None,
                         w.draft_tokens.numpy(), w.u_accept.numpy(), w.u_final.numpy(), T, rows=rows)


def flag_budget(w, ref, rows=None):
    """Upper tail of the number of rows the oracle may flag, from the exact
    flag probabilities of each row.  Over a uniform u', a draw from weights w
    is flagged when u' lies within 1e-6 of either end of the chosen token's
    CDF interval [C_{v-1}, C_v) / Z, with probability sum_v min(w_v / Z, 2e-6);
    each evaluated acceptance adds at most 2e-6 (|u - p/q| < 1e-6).  A
    threshold or operand gone wrong in the oracle flags far more rows than
    this bound allows."""
    eps = oracle.spec_oracle.NEAR_TIE
    T = w.temperature
    B, K, _ = w.shape
    rows = range(B) if rows is None else rows
    e = 0.0
    for i, b in enumerate(rows):
        n = int(ref.n_accepted[i])
        zt = synth.f64(w.target[b])
        p = oracle.softmax_t(zt[n], T)
        if n < K:
            r = oracle.residual(p, oracle.softmax_t(synth.f64(w.draft[b, n]), T))
            wts = r if r.sum() > 0 else p
        else:
            wts = p
        e += float(np.minimum(wts / wts.sum(), 2 * eps).sum()) + 2 * eps * (min(n + 1, K))
    return e + 4.0 * np.sqrt(e) + 3.0


def assert_verify(out, ref, rows=None, check_alpha=True):
    tok = out.tokens.cpu().numpy()
    n = out.n_accepted.cpu().numpy()
    if rows is not None:
        tok, n = tok[rows], n[rows]
    ok = ~ref.flagged
    bad = np.nonzero(ok & ((tok != ref.tokens).any(axis=1) | (n != ref.n_accepted)))[0]
    assert bad.size == 0, f"rows {bad[:10]}: gpu {tok[bad[:3]]} n {n[bad[:3]]} vs oracle {ref.tokens[bad[:3]]} " \
                          f"n {ref.n_accepted[bad[:3]]}"
    if check_alpha and out.alpha is not None:
        a = out.alpha.cpu().numpy()
        if rows is not None:
            a = a[rows]
        np.testing.assert_allclose(a, ref.alpha, rtol=RTOL, atol=ATOL)
    return int(ref.flagged.sum())


# ---------------------------------------------------------------------------
# the seeded small case: 1000 calls of B=1, K=4, V=1024 fp32
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kernel", [0, 2], ids=["automatic", "two_pass"])
def test_small_case_1000_seeded_calls(ssv, kernel):
    flagged = 0
    hist = np.zeros(5, dtype=np.int64)
    ssv.set_kernel_override(kernel)
    try:
        for seed in range(1000):
            w = synth.small(seed=seed)
            out = ssv.verify(*to_dev(w), w.temperature)
            ref = oracle_verify(w)
            flagged += assert_verify(out, ref)
            assert int(out.status.item()) == 0
            hist[int(ref.n_accepted[0])] += 1
    finally:
        ssv.set_kernel_override(0)
    print(f"flagged rows: {flagged} / 1000; accepted-count histogram {hist.tolist()}")
    assert flagged < 10


# ---------------------------------------------------------------------------
# shapes spanning several tiles, ragged tails and degenerate cases
# ---------------------------------------------------------------------------

CASES = [
    # B, K, V, dtype, T
    (3, 2, 1, torch.float32, 1.0),         # a one-token vocabulary
    (2, 3, 7, torch.bfloat16, 0.7),        # V smaller than one vector, ragged rows
    (4, 3, 5003, torch.bfloat16, 1.0),     # ragged V: element-wise staging
    (4, 3, 5003, torch.float32, 1.3),
    (4, 3, 4096, torch.float32, 2.0),      # aligned fp32
    (2, 0, 1000, torch.bfloat16, 1.0),     # K = 0: plain sampling of the bonus row
    (5, 16, 3000, torch.bfloat16, 1.0),    # long draft block
    (2, 33, 520, torch.float32, 0.9),      # K + 1 above one warp
    (6, 4, 40000, torch.bfloat16, 0.5),    # several CTAs per cluster
    (3, 4, 40000, torch.bfloat16, 0.0),    # greedy
    (3, 4, 40001, torch.float32, 0.0),     # greedy, ragged
    (7, 2, 131072, torch.bfloat16, 1.0),   # a power-of-two vocabulary
]


@pytest.mark.parametrize("B,K,V,dtype,T", CASES)
def test_shapes_against_oracle(ssv, B, K, V, dtype, T):
    w = synth.gaussian(B, K, V, sigma=2.0, noise=0.6, dtype=dtype, temperature=T, seed=B * 1000 + K * 10 + V)
    out = ssv.verify(*to_dev(w), w.temperature)
    torch.cuda.synchronize()
    ref = oracle_verify(w)
    assert_verify(out, ref)
    assert int(out.status.item()) == 0
    # tokens after the emitted one are -1, emitted ones are valid ids
    tok = out.tokens.cpu().numpy()
    n = out.n_accepted.cpu().numpy()
    for b in range(B):
        assert (tok[b, : n[b] + 1] >= 0).all() and (tok[b, : n[b] + 1] < V).all()
        assert (tok[b, n[b] + 1:] == -1).all()


@pytest.mark.parametrize("S,nst", [(1, 2), (2, 1), (3, 2), (4, 1), (8, 2), (12, 1), (16, 2)])
def test_launch_shapes_agree(ssv, S, nst):
    w = synth.gaussian(6, 3, 24000, sigma=2.0, noise=0.6, dtype=torch.bfloat16, temperature=1.0, seed=77)
    ssv.set_launch_override(S, nst)
    try:
        assert ssv.launch_shape(torch.bfloat16, 6 * 4, 24000)[0] == S
        out = ssv.verify(*to_dev(w), w.temperature)
        torch.cuda.synchronize()
    finally:
        ssv.set_launch_override(0, 0)
    assert_verify(out, oracle_verify(w))


def test_row_groups_with_draw_skip_against_oracle(ssv):
    """More rows than clusters: rows run in groups, position-major inside a
    group, and units skip draws that an earlier rejection makes unused.  Every
    row against the oracle (tokens, counts and alpha of skipped rejections),
    with a partial last group."""
    B, K, V = 230, 3, 6000
    w = synth.gaussian(B, K, V, sigma=2.0, noise=1.0, dtype=torch.float32, temperature=1.0, seed=4545)
    ssv.set_launch_override(16, 1)
    try:
        G = ssv.launch_shape(torch.float32, B * (K + 1), V)[3]
        assert B > G and B % G != 0, G
        out = ssv.verify(*to_dev(w), w.temperature)
        torch.cuda.synchronize()
    finally:
        ssv.set_launch_override(0, 0)
    ref = oracle_verify(w)
    assert_verify(out, ref)
    assert (ref.n_accepted < K - 1).sum() > 20  # many rows with positions after the first rejection


def test_greedy_ties_take_smallest_index(ssv):
    B, K, V = 4, 3, 2048
    zt = torch.zeros((B, K + 1, V), dtype=torch.bfloat16)
    # several equal maxima per row, including across CTA slices
    for b in range(B):
        for k in range(K + 1):
            idx = torch.tensor([100 + 37 * b + k, 1500, 2047, 900])
            zt[b, k, idx] = 3.0
    zd = zt[:, :K].clone()
    y = torch.full((B, K), 100, dtype=torch.int32)
    y[:, 0] = torch.tensor([100 + 37 * b for b in range(B)], dtype=torch.int32)
    out = ssv.verify(zt.to(DEV), zd.to(DEV), y.to(DEV), None, None, 0.0)
    torch.cuda.synchronize()
    ref = oracle.verify(zt.double().numpy(), zd.double().numpy(), y.numpy(), np.zeros((B, K)), np.zeros(B), 0.0)
    assert (out.tokens.cpu().numpy() == ref.tokens).all()
    assert (out.n_accepted.cpu().numpy() == ref.n_accepted).all()


# ---------------------------------------------------------------------------
# full-size workloads
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T", [0.0, 0.7, 1.0])
def test_entropy_mix_full_size(ssv, T):
    w = synth.entropy_mix(seed=1235, temperature=T)
    out = ssv.verify(*to_dev(w), w.temperature)
    torch.cuda.synchronize()
    ref = oracle_verify(w)
    flagged = assert_verify(out, ref)
    budget = flag_budget(w, ref) if T > 0 else 0
    print(f"T={T}: flagged rows {flagged} / {w.shape[0]} (bound {budget:.1f}), mean accepted "
          f"{ref.n_accepted.mean():.3f}")
    assert flagged <= budget, (flagged, budget)
    assert int(out.status.item()) == 0


def test_zipf_full_size(ssv):
    """The Zipf workload (B=128, K=7, V=129280 bf16, T=1) runs the row-grouped
    kernel with draw skipping: every row against the oracle."""
    w = synth.zipf(seed=1236)
    out = ssv.verify(*to_dev(w), w.temperature)
    torch.cuda.synchronize()
    assert int(out.status.item()) == 0
    B, K, V = w.shape
    n = out.n_accepted.cpu().numpy()
    a = out.alpha.cpu().numpy()
    same = np.setdiff1d(np.arange(B), w.low_rows)
    # draft == target bitwise: every draft accepted, alpha 1
    assert (n[same] == K).all()
    np.testing.assert_allclose(a[same], 1.0, rtol=0, atol=2e-6)
    ref = oracle_verify(w)
    flagged = assert_verify(out, ref)
    budget = flag_budget(w, ref)
    print(f"zipf: flagged rows {flagged} / {B} (bound {budget:.1f})")
    assert flagged <= budget, (flagged, budget)


def test_sweep_points_sampled_rows(ssv):
    """Points of the B x K grid at V=151936: every row up to B=64, sampled rows
    at B=256."""
    for B, K in ((1, 1), (8, 2), (64, 7), (64, 16), (256, 4)):
        w = synth.sweep(B, K, seed=1238 + B + K)
        out = ssv.verify(*to_dev(w), w.temperature)
        torch.cuda.synchronize()
        rows = list(range(B)) if B <= 64 else sorted(set(range(0, B, 8)) | {B - 1})
        ref = oracle_verify(w, rows=rows)
        flagged = assert_verify(out, ref, rows=rows)
        budget = flag_budget(w, ref, rows)
        assert flagged <= budget, (B, K, flagged, budget)
        n = out.n_accepted.cpu().numpy()
        assert (n >= 0).all() and (n <= K).all()
        del w, out
        torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# overlap statistics
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("B,K,V,dtype,T", [(4, 5, 30000, torch.bfloat16, 1.0), (3, 2, 999, torch.float32, 0.6),
                                           (5, 3, 20000, torch.bfloat16, 0.0)])
def test_overlap_against_oracle(ssv, B, K, V, dtype, T):
    w = synth.gaussian(B, K, V, sigma=2.0, noise=0.5, dtype=dtype, temperature=max(T, 1.0), seed=B + K + V,
                       draft_tokens=False)
    t = w.target.to(DEV)  # [B, K+1, V]: the verify layout, first K positions used
    o = ssv.overlap(t, w.draft.to(DEV), T)
    torch.cuda.synchronize()
    ref = oracle.overlap_stats(synth.f64(w.target[:, :K]), synth.f64(w.draft), T)
    np.testing.assert_allclose(o.alpha.cpu().numpy(), ref.alpha, rtol=RTOL, atol=ATOL)
    np.testing.assert_allclose(o.tv.cpu().numpy(), ref.tv, rtol=RTOL, atol=ATOL)
    np.testing.assert_allclose(o.prefix_survival.cpu().numpy(), ref.prefix_survival, rtol=RTOL, atol=ATOL)
    np.testing.assert_allclose(o.expected_accepted.cpu().numpy(), ref.expected_accepted, rtol=RTOL, atol=ATOL)


# ---------------------------------------------------------------------------
# E2E-TV loss and gradient
# ---------------------------------------------------------------------------

def _check_grad(g_gpu, w, T, scale, rows):
    rg, amb = oracle.e2e_tv_grad(synth.f64(w.target), synth.f64(w.draft), T, grad_scale=scale, rows=rows)
    gg = g_gpu[rows]
    err = np.abs(gg - rg)
    tol = ATOL + RTOL * np.abs(rg)
    bad = (err > tol) & ~amb
    assert not bad.any(), f"{bad.sum()} gradient elements off, worst {err[bad].max()}"
    rel = np.linalg.norm(gg - rg) / max(np.linalg.norm(rg), 1e-30)
    assert rel < 1e-4, rel
    return int(amb.sum())


@pytest.mark.parametrize("B,K,V,dtype,T", [(3, 4, 3000, torch.float32, 1.0), (4, 7, 20011, torch.bfloat16, 0.8),
                                           (2, 1, 50000, torch.bfloat16, 1.0)])
def test_e2e_small_against_oracle(ssv, B, K, V, dtype, T):
    w = synth.gaussian(B, K, V, sigma=2.0, noise=0.5, dtype=dtype, temperature=T, seed=7 * B + K,
                       bonus=False, draft_tokens=False)
    e = ssv.e2e_tv_fwd_bwd(w.target.to(DEV), w.draft.to(DEV), w.temperature, grad_scale=-1.0)
    torch.cuda.synchronize()
    L, a = oracle.e2e_tv_loss(synth.f64(w.target), synth.f64(w.draft), w.temperature)
    assert abs(float(e.loss.item()) - L) <= ATOL + RTOL * abs(L)
    np.testing.assert_allclose(e.alpha.cpu().numpy(), a, rtol=RTOL, atol=ATOL)
    _check_grad(e.grad.cpu().numpy(), w, w.temperature, -1.0, list(range(B)))


def test_e2e_full_size(ssv):
    w = synth.e2e(seed=1237)
    B, K, V = w.shape
    e = ssv.e2e_tv_fwd_bwd(w.target.to(DEV), w.draft.to(DEV), 1.0, grad_scale=1.0)
    torch.cuda.synchronize()
    assert int(e.status.item()) == 0
    L, a = oracle.e2e_tv_loss(synth.f64(w.target), synth.f64(w.draft), 1.0)
    assert abs(float(e.loss.item()) - L) <= ATOL + RTOL * abs(L)
    np.testing.assert_allclose(e.alpha.cpu().numpy(), a, rtol=RTOL, atol=ATOL)
    g = e.grad.cpu().numpy()
    # the gradient of each softmax row sums to zero
    assert np.abs(g.sum(axis=2)).max() < 1e-6
    rows = list(range(0, B, 8))  # 32 of the 256 rows, element by element
    amb = _check_grad(g, w, 1.0, 1.0, rows)
    print(f"ambiguous indicator elements in {len(rows)} rows: {amb}")


# ---------------------------------------------------------------------------
# the output distribution equals p (1e6 rows in one call)
# ---------------------------------------------------------------------------

def test_distribution_chi_square_1e6_rows(ssv):
    from scipy.stats import chisquare
    rng = np.random.default_rng(99)
    N, K, V = 1_000_000, 3, 5
    zt1 = rng.standard_normal((K + 1, V)) * 1.2
    zd1 = rng.standard_normal((K, V)) * 1.2
    zt1 = zt1.astype(np.float32).astype(np.float64)
    zd1 = zd1.astype(np.float32).astype(np.float64)
    p = [oracle.softmax_t(zt1[k], 1.0) for k in range(K + 1)]
    q = [oracle.softmax_t(zd1[k], 1.0) for k in range(K)]
    cq = [np.cumsum(x) for x in q]
    y = np.stack([np.minimum(np.searchsorted(cq[k], rng.random(N), side="right"), V - 1) for k in range(K)], 1)
    ua = rng.random((N, K), dtype=np.float32)
    uf = rng.random(N, dtype=np.float32)
    t = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(zt1, (N, K + 1, V)), dtype=np.float32)).to(DEV)
    d = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(zd1, (N, K, V)), dtype=np.float32)).to(DEV)
    out = ssv.verify(t, d, torch.from_numpy(y.astype(np.int32)).to(DEV), torch.from_numpy(ua).to(DEV),
                     torch.from_numpy(uf).to(DEV), 1.0)
    torch.cuda.synchronize()
    tok = out.tokens.cpu().numpy()
    n = out.n_accepted.cpu().numpy()

    def pval(counts, probs):
        return chisquare(counts, np.asarray(probs) * counts.sum()).pvalue

    assert pval(np.bincount(tok[:, 0], minlength=V), p[0]) > 1e-3
    for j in range(1, K + 1):
        sel = n >= j
        assert pval(np.bincount(tok[sel, j], minlength=V), p[j]) > 1e-3
    alpha = [oracle.overlap(p[k], q[k]) for k in range(K)]
    surv = [1.0] + oracle.prefix_survival(alpha)
    pn = [surv[j] - (surv[j + 1] if j < K else 0.0) for j in range(K + 1)]
    assert pval(np.bincount(n, minlength=K + 1), pn) > 1e-3
    # and every row agrees with the oracle's decisions on a sample
    sample = rng.choice(N, 2000, replace=False)
    p_rows = np.asarray(p)
    q_rows = np.asarray(q)
    for i in sample:
        toks, nn, a_near, c_near, _ = oracle.accept_and_correct(p_rows, q_rows, y[i], ua[i].astype(np.float64),
                                                                float(uf[i]))
        if not (a_near or c_near):
            assert list(tok[i]) == toks and n[i] == nn


# ---------------------------------------------------------------------------
# edge cases and the device status word
# ---------------------------------------------------------------------------

def test_identical_and_disjoint_logits(ssv):
    B, K, V = 8, 4, 3000
    w = synth.gaussian(B, K, V, sigma=2.0, noise=0.0, dtype=torch.bfloat16, temperature=1.0, seed=5)
    out = ssv.verify(*to_dev(w), 1.0)
    torch.cuda.synchronize()
    assert (out.n_accepted.cpu().numpy() == K).all()
    np.testing.assert_allclose(out.alpha.cpu().numpy(), 1.0, atol=2e-6)
    assert_verify(out, oracle_verify(w))
    # disjoint supports: the draft puts all its mass where p has none
    zt = torch.full((B, K + 1, V), -1e4, dtype=torch.float32)
    zd = torch.full((B, K, V), -1e4, dtype=torch.float32)
    zt[:, :, : V // 2] = 0.0
    zd[:, :, V // 2:] = 0.0
    y = torch.full((B, K), V - 1, dtype=torch.int32)
    ua = torch.rand((B, K), dtype=torch.float32)
    uf = torch.rand((B,), dtype=torch.float32)
    out = ssv.verify(zt.to(DEV), zd.to(DEV), y.to(DEV), ua.to(DEV), uf.to(DEV), 1.0)
    torch.cuda.synchronize()
    assert (out.n_accepted.cpu().numpy() == 0).all()
    tok0 = out.tokens.cpu().numpy()[:, 0]
    assert ((tok0 >= 0) & (tok0 < V // 2)).all()
    np.testing.assert_allclose(out.alpha.cpu().numpy(), 0.0, atol=1e-6)


@pytest.fixture(params=[1, 2], ids=["single_read", "two_pass"])
def sweep_kernel(ssv, request):
    """Runs a test with each sweep forced (the automatic choice takes the
    single-read sweep at these sizes)."""
    ssv.set_kernel_override(request.param)
    yield request.param
    ssv.set_kernel_override(0)


def test_status_bits(ssv, sweep_kernel):
    B, K, V = 3, 2, 1000
    w = synth.gaussian(B, K, V, sigma=1.0, noise=0.5, dtype=torch.float32, temperature=1.0, seed=6)
    t, d, y, ua, uf = to_dev(w)
    y2 = y.clone()
    y2[1, 0] = V + 5
    out = ssv.verify(t, d, y2, ua, uf, 1.0)
    torch.cuda.synchronize()
    assert int(out.status.item()) & ssv.DEV_BAD_TOKEN
    assert int(out.n_accepted[1].item()) == 0
    t2 = t.clone()
    t2[2, 1, 17] = float("nan")
    out = ssv.verify(t2, d, y, ua, uf, 1.0)
    torch.cuda.synchronize()
    assert int(out.status.item()) & ssv.DEV_BAD_LOGITS
    ua2 = ua.clone()
    ua2[0, 0] = 1.5
    out = ssv.verify(t, d, y, ua2, uf, 1.0)
    torch.cuda.synchronize()
    assert int(out.status.item()) & ssv.DEV_BAD_UNIFORM


def test_empty_residual_reported_for_the_emitted_position(ssv, sweep_kernel):
    """EMPTY_RESIDUAL is raised only by the rejection a row emits (the
    oracle's ``residual_empty``), whatever later positions hold."""
    B, K, V = 2, 3, 1000
    w = synth.gaussian(B, K, V, sigma=1.0, noise=0.5, dtype=torch.float32, temperature=1.0, seed=8)
    t, d, y, ua, uf = to_dev(w)
    d2 = d.clone()
    d2[:, 2] = t[:, 2]   # position 2: q = p
    d2[0, 1] = t[0, 1]   # row 0, position 1: q = p
    y2 = y.clone()
    ua2 = ua.clone()
    ua2[0, 0] = 0.0      # row 0: position 0 accepted
    y2[0, 1] = V + 1     # row 0: rejected at 1 with an empty residual: drawn from p_1
    y2[1, 0] = V + 1     # row 1: rejected at 0, residual not empty
    y2[1, 2] = V + 1     # row 1: position 2 empty but never emitted
    both = ssv.verify(t, d2, y2, ua2, uf, 1.0)
    row1 = ssv.verify(t[1:].contiguous(), d2[1:].contiguous(), y2[1:].contiguous(), ua2[1:].contiguous(),
                      uf[1:].contiguous(), 1.0)
    torch.cuda.synchronize()
    assert int(both.status.item()) == ssv.DEV_BAD_TOKEN | ssv.DEV_EMPTY_RESIDUAL
    assert int(row1.status.item()) == ssv.DEV_BAD_TOKEN
    assert both.n_accepted.cpu().tolist() == [1, 0]
    p01 = oracle.softmax_t(synth.f64(w.target[0, 1]), 1.0)
    v, _ = oracle.inverse_cdf(p01, float(w.u_final[0]))
    assert int(both.tokens[0, 1]) == v
    zt, zd = synth.f64(w.target[1, 0]), synth.f64(w.draft[1, 0])
    rho = oracle.residual(oracle.softmax_t(zt, 1.0), oracle.softmax_t(zd, 1.0))
    v1, _ = oracle.inverse_cdf(rho, float(w.u_final[1]))
    assert int(both.tokens[1, 0]) == v1 == int(row1.tokens[0, 0])


def test_empty_batch_and_invalid_args(ssv):
    z = torch.zeros((0, 3, 10), device=DEV)
    out = ssv.verify(z, torch.zeros((0, 2, 10), device=DEV), torch.zeros((0, 2), dtype=torch.int32, device=DEV),
                     torch.zeros((0, 2), device=DEV), torch.zeros((0,), device=DEV), 1.0)
    assert out.tokens.shape == (0, 3)
    with pytest.raises(ssv.SpecError):
        ssv.e2e_tv_fwd_bwd(torch.zeros((1, 2, 10), device=DEV), torch.zeros((1, 2, 10), device=DEV), 0.0)


def test_deterministic_and_workspace_left_zero(ssv):
    w = synth.gaussian(16, 5, 60000, sigma=2.0, noise=0.7, dtype=torch.bfloat16, temperature=1.0, seed=9)
    args = to_dev(w)
    L = ssv.lib()
    nbytes = max(L.spec_verify_workspace_bytes(16, 5, 60000), L.spec_e2e_tv_workspace_bytes(16, 5, 60000))
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
    a = ssv.verify(*args, 1.0, workspace=ws)
    b = ssv.verify(*args, 1.0, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a.tokens, b.tokens) and torch.equal(a.n_accepted, b.n_accepted)
    assert torch.equal(a.alpha, b.alpha)
    # every call leaves the whole workspace zero-filled
    assert int(ws.count_nonzero().item()) == 0
    # shared between entry points and shapes without re-zeroing
    e = ssv.e2e_tv_fwd_bwd(args[0], args[1], 1.0, K=5, workspace=ws)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero().item()) == 0
    c = ssv.verify(args[0][:3].contiguous(), args[1][:3].contiguous(), args[2][:3].contiguous(),
                   args[3][:3].contiguous(), args[4][:3].contiguous(), 1.0, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(c.tokens, a.tokens[:3]) and int(ws.count_nonzero().item()) == 0
    assert np.isfinite(float(e.loss.item()))


def test_unaligned_rows_match_aligned(ssv):
    """Rows off 16-byte boundaries take the single-read sweep, aligned rows
    the two-pass sweep: both match the oracle and each other within the
    parity bar."""
    B, K, V = 3, 3, 4096
    w = synth.gaussian(B, K, V, sigma=2.0, noise=0.6, dtype=torch.bfloat16, temperature=1.0, seed=12)
    t, d, y, ua, uf = to_dev(w)
    ref = ssv.verify(t, d, y, ua, uf, 1.0)
    # same data at an address 2 bytes off a 16-byte boundary
    bt = torch.empty(t.numel() + 8, dtype=t.dtype, device=DEV)
    bd = torch.empty(d.numel() + 8, dtype=d.dtype, device=DEV)
    t2 = bt[1:1 + t.numel()].view(t.shape)
    d2 = bd[1:1 + d.numel()].view(d.shape)
    t2.copy_(t)
    d2.copy_(d)
    out = ssv.verify(t2, d2, y, ua, uf, 1.0)
    torch.cuda.synchronize()
    orc = oracle_verify(w)
    assert_verify(out, orc)
    assert_verify(ref, orc)
    ok = ~orc.flagged
    assert (out.tokens.cpu().numpy()[ok] == ref.tokens.cpu().numpy()[ok]).all()
    np.testing.assert_allclose(out.alpha.cpu().numpy(), ref.alpha.cpu().numpy(), rtol=RTOL, atol=ATOL)


def test_host_verifier_round_trip(ssv):
    w = synth.gaussian(4, 3, 8192, sigma=2.0, noise=0.6, dtype=torch.bfloat16, temperature=1.0, seed=13)
    hv = ssv.HostVerifier(4, 3, 8192, dtype=torch.bfloat16)
    pin = lambda x: x.pin_memory()  # noqa: E731
    tok = torch.empty((4, 4), dtype=torch.int32).pin_memory()
    n = torch.empty((4,), dtype=torch.int32).pin_memory()
    a = torch.empty((4, 3), dtype=torch.float32).pin_memory()
    hv.run(pin(w.target), pin(w.draft), pin(w.draft_tokens), pin(w.u_accept), pin(w.u_final), 1.0, tok, n, a)
    ref = oracle_verify(w)
    ok = ~ref.flagged
    assert (tok.numpy()[ok] == ref.tokens[ok]).all() and (n.numpy()[ok] == ref.n_accepted[ok]).all()
