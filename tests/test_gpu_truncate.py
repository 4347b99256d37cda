"""GPU parity of top-k / top-p truncation against the fp64 oracle, and of a
verify step on truncated target and draft logits.

Bar: the kept set (which logits stay finite) is bit-exact on every row the
oracle does not flag as a near top-p tie (preceding mass within 1e-5 of
top_p); on a flagged row it lies between the oracle's kept sets for
top_p - 1e-5 and top_p + 1e-5.  Kept logits are copied bit for bit.
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


def _check_rows(z_in, z_out, T, k, p, rows=None):
    zi = synth.f64(z_in.reshape(-1, z_in.shape[-1]).cpu())
    zo = z_out.reshape(-1, z_out.shape[-1]).cpu()
    rows = range(zi.shape[0]) if rows is None else rows
    flagged = 0
    for r in rows:
        want, near = oracle.truncate_logits(zi[r], T, k, p)
        got = synth.f64(zo[r])
        keep_g = np.isfinite(got)
        assert (got[keep_g] == zi[r][keep_g]).all()
        if near:
            flagged += 1
            lo = np.isfinite(oracle.truncate_logits(zi[r], T, k, p - oracle.NEAR_TRUNC)[0])
            hi = np.isfinite(oracle.truncate_logits(zi[r], T, k, min(p + oracle.NEAR_TRUNC, 1.0))[0])
            assert (lo <= keep_g).all() and (keep_g <= hi).all(), f"row {r}: cut outside the near-tie bracket"
            continue
        keep_w = np.isfinite(want)
        bad = np.nonzero(keep_w != keep_g)[0]
        assert bad.size == 0, f"row {r}: {bad.size} tokens differ, first {bad[:5]}, kept {keep_g.sum()} vs {keep_w.sum()}"
        assert (got[keep_g] == zi[r][keep_g]).all()
    return flagged


CASES = [
    # V, dtype, T, top_k, top_p
    (4096, torch.bfloat16, 1.0, 50, 1.0),
    (4096, torch.bfloat16, 1.0, 0, 0.9),
    (4096, torch.bfloat16, 0.7, 40, 0.8),
    (20011, torch.bfloat16, 1.3, 1, 1.0),      # unaligned rows
    (20011, torch.bfloat16, 1.0, 500, 0.95),
    (1001, torch.float32, 1.0, 10, 0.5),       # unaligned fp32
    (3000, torch.float32, 0.8, 2999, 0.99),
    (3000, torch.float32, 1.0, 0, 0.05),
    (3000, torch.float32, 1.0, 3000, 1.0),     # nothing to do: a copy
]


@pytest.mark.parametrize("V,dtype,T,k,p", CASES)
def test_rows_against_oracle(ssv, V, dtype, T, k, p):
    g = torch.Generator().manual_seed(V + k)
    rows = 12
    sig = torch.tensor([0.5, 1.0, 2.0, 4.0]).repeat(3)[:, None]
    z = torch.randn(rows, V, generator=g) * sig
    z[::3] = torch.round(z[::3] * 4) / 4  # many exact ties
    z = z.to(dtype)
    zd = z.to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = ssv.truncate_logits(zd, T, k, p, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    flagged = _check_rows(z, out, T, k, p)
    print(f"near top-p ties: {flagged} of {rows} rows")
    # in place gives the same bits
    zz = zd.clone()
    ssv.truncate_logits(zz, T, k, p, out=zz)
    torch.cuda.synchronize()
    assert torch.equal(zz, out)


def test_ties_at_both_cuts(ssv):
    """Equal logits straddling the top-k and the top-p boundaries keep the
    smallest indices."""
    V = 2048
    z = torch.full((2, V), -3.0)
    z[:, 100:110] = 2.0
    z[:, 500:540] = 1.0   # ties across the top-k cut below
    z[:, 7] = 4.0
    zb = z.to(torch.bfloat16)
    out = ssv.truncate_logits(zb.to(DEV), 1.0, 30, 0.93)
    out2 = ssv.truncate_logits(zb.to(DEV), 1.0, 30, 1.0)
    torch.cuda.synchronize()
    k2 = torch.isfinite(out2[0].float()).nonzero().flatten().tolist()
    assert k2 == [7] + list(range(100, 110)) + list(range(500, 519))
    _check_rows(zb, out, 1.0, 30, 0.93)


@pytest.mark.parametrize("k,p", [(50, 1.0), (3000, 1.0), (0, 0.9), (50, 0.9), (3000, 0.95), (8000, 0.999)])
def test_value_histogram_limits(ssv, k, p):
    """bf16 rows at the limits of the one-pass value histogram, each against
    the oracle: dropped (-inf) logits, values at or above 2^16, zeros beside
    a small maximum, a top-k cut among -inf, ties, zeros beside a large
    maximum, mostly tiny values, and a wide range."""
    V = 8192
    g = torch.Generator().manual_seed(5)
    z = torch.randn(8, V, generator=g) * 2
    z[0, ::3] = -float("inf")                     # an already truncated row
    z[1, :100] = 70000.0                          # at and above 2^16
    z[1, 100:200] = 65536.0
    z[2] = torch.log_softmax(z[2], 0)             # log-probabilities: maximum near 0
    z[2, ::5] = 0.0                               # zeros beside it
    z[3, 40:] = -float("inf")                     # fewer finite logits than some top_k
    z[4] = torch.round(z[4] * 4) / 4              # heavy ties
    z[5, ::2] = 0.0                               # zeros beside a maximum above 2
    z[6] = torch.randn(V, generator=g) * 1e-6     # magnitudes around 2^-20
    z[7] = z[7] * 300                             # a wide range
    zb = z.to(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = ssv.truncate_logits(zb.to(DEV), 1.0, k, p, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _check_rows(zb, out, 1.0, k, p)
    if p == 1.0:  # top-k of a top-k row keeps it
        again = ssv.truncate_logits(out, 1.0, k, 1.0)
        torch.cuda.synchronize()
        assert torch.equal(again, out)


def test_topk_exactly_k_pass_the_first_bound(ssv):
    """A row whose k largest logits are each the largest of one lane's first
    vectors, everything else far below: the candidate path's first bound
    lets exactly k elements through, and only those may stay."""
    V, k = 32768, 50                      # 4096 vectors of 8 bf16; 256 per warp
    g = torch.Generator().manual_seed(31)
    z = torch.randn(2, V, generator=g)
    pos = [(w * 256 + lane) * 8 for w in (0, 1) for lane in range(32)][:k]
    z[0, pos] = 100.0 + torch.arange(k, dtype=torch.float32)
    z[1, pos] = 100.0                     # the same with all k tied
    zb = z.to(torch.bfloat16)
    out = ssv.truncate_logits(zb.to(DEV), 1.0, k, 1.0)
    torch.cuda.synchronize()
    kept = torch.isfinite(out.float().cpu())
    assert kept[0].nonzero().flatten().tolist() == pos
    assert kept[1].nonzero().flatten().tolist() == pos
    _check_rows(zb, out, 1.0, k, 1.0)


def test_full_size_verify_batch_and_verify_on_truncated(ssv):
    """The verify batch (B=32, K=4, V=151936): truncate target and draft
    identically, draw the drafted tokens from the truncated q, verify, and
    compare tokens with the oracle run on the truncated logits."""
    w = synth.entropy_mix(seed=2024)
    B, K, V = w.shape
    T, k, p = 1.0, 50, 0.9
    t = ssv.truncate_logits(w.target.to(DEV), T, k, p)
    d = ssv.truncate_logits(w.draft.to(DEV), T, k, p)
    torch.cuda.synchronize()
    ft = _check_rows(w.target, t, T, k, p)
    fd = _check_rows(w.draft, d, T, k, p)
    print(f"near top-p ties: {ft} target rows, {fd} draft rows")
    # drafted tokens from the truncated draft (Gumbel-max on finite logits)
    g = torch.Generator().manual_seed(77)
    dc = d.float().cpu()
    gum = -torch.log(-torch.log(torch.rand(dc.shape, generator=g).clamp_min(1e-20)))
    y = torch.argmax(dc / T + gum, dim=-1).to(torch.int32)
    assert torch.isfinite(dc.gather(2, y.long()[..., None])).all()
    out = ssv.verify(t, d, y.to(DEV), w.u_accept.to(DEV), w.u_final.to(DEV), T)
    torch.cuda.synchronize()
    assert int(out.status.item()) == 0
    ref = oracle.verify(synth.f64(t.cpu()), synth.f64(d.cpu()), y.numpy(), w.u_accept.numpy(),
                        w.u_final.numpy(), T)
    tok = out.tokens.cpu().numpy()
    n = out.n_accepted.cpu().numpy()
    ok = ~ref.flagged
    assert ((tok == ref.tokens).all(axis=1) | ~ok).all()
    assert ((n == ref.n_accepted) | ~ok).all()
    np.testing.assert_allclose(out.alpha.cpu().numpy(), ref.alpha, rtol=1e-4, atol=1e-6)
    # every emitted token lies in the target's kept set
    tf = torch.isfinite(t.float().cpu())
    for b in range(B):
        for j in range(int(n[b]) + 1):
            assert tf[b, j, int(tok[b, j])]


def test_bad_rows_copied_and_flagged(ssv):
    z = torch.randn(3, 1024)
    z[1, 5] = float("nan")
    z[2, :] = -float("inf")
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = ssv.truncate_logits(z.to(DEV), 1.0, 10, 0.9, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & ssv.DEV_BAD_LOGITS
    o = out.cpu()
    assert torch.isfinite(o[0]).sum() <= 10
    assert torch.equal(torch.isnan(o[1]), torch.isnan(z[1])) and torch.equal(o[1][~torch.isnan(z[1])],
                                                                          z[1][~torch.isnan(z[1])])
    assert torch.equal(o[2], z[2])


def test_invalid_arguments(ssv):
    x = torch.randn(2, 64, device=DEV)
    for kw in (dict(top_k=-1), dict(top_p=0.0), dict(top_p=1.5)):
        with pytest.raises(ssv.SpecError):
            ssv.truncate_logits(x, 1.0, **kw)
    with pytest.raises(ssv.SpecError):
        ssv.truncate_logits(x, 0.0, 0, 0.9)  # top-p needs T > 0
    ssv.truncate_logits(x, 0.0, 5, 1.0)      # top-k alone does not
    # an output that overlaps the input without being it is refused
    import ctypes
    buf = torch.randn(4 * 64, device=DEV)
    rc = ssv.lib().spec_truncate_logits(ctypes.c_void_p(buf.data_ptr()), ctypes.c_void_p(buf.data_ptr() + 32), 0,
                                        2, 64, 1.0, 3, 1.0, None, None)
    assert rc == ssv.SPEC_ERR_INVALID_ARG
