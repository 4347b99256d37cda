"""GPU parity of the ragged verify (a length of its own per row, flattened
tensors) against the fp64 oracle run row by row with that row's length.

Bar: as for the fixed-length verify -- tokens and accepted counts bit-exact
outside the oracle's near-tie flags; alpha within 1e-4 relative + 1e-6.
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


def flatten(w, lengths):
    """Row b keeps drafted positions 0..l_b-1 and its target position l_b as
    the bonus distribution."""
    B = w.shape[0]
    off = np.zeros(B + 1, dtype=np.int32)
    off[1:] = np.cumsum(np.asarray(lengths) + 1)
    tg = torch.cat([w.target[b, : l + 1] for b, l in enumerate(lengths)])
    dr = [w.draft[b, :l] for b, l in enumerate(lengths)]
    nd = int(sum(lengths))
    dr = torch.cat(dr) if nd else None
    tok = torch.cat([w.draft_tokens[b, :l] for b, l in enumerate(lengths)])
    ua = torch.cat([w.u_accept[b, :l] for b, l in enumerate(lengths)])
    return off, tg, dr, tok, ua


def run(ssv, w, lengths, T):
    off, tg, dr, tok, ua = flatten(w, lengths)
    out = ssv.verify_ragged(tg.contiguous().to(DEV), None if dr is None else dr.contiguous().to(DEV),
                            torch.from_numpy(off).to(DEV), tok.contiguous().to(DEV), ua.contiguous().to(DEV),
                            w.u_final.to(DEV), T)
    torch.cuda.synchronize()
    return off, out


def check(w, lengths, T, off, out):
    tok = out.tokens.cpu().numpy()
    n = out.n_accepted.cpu().numpy()
    al = out.alpha.cpu().numpy() if out.alpha is not None else None
    flagged = 0
    for b, l in enumerate(lengths):
        ref = oracle.verify(synth.f64(w.target[b: b + 1, : l + 1]), synth.f64(w.draft[b: b + 1, :l]),
                            w.draft_tokens[b: b + 1, :l].numpy(), w.u_accept[b: b + 1, :l].numpy(),
                            w.u_final[b: b + 1].numpy(), T)
        if ref.flagged[0]:
            flagged += 1
            continue
        assert n[b] == ref.n_accepted[0], (b, l)
        np.testing.assert_array_equal(tok[off[b]: off[b + 1]], ref.tokens[0], err_msg=f"row {b}")
        if l and al is not None:
            d0 = off[b] - b
            np.testing.assert_allclose(al[d0: d0 + l], ref.alpha[0], rtol=1e-4, atol=1e-6)
    return flagged


@pytest.mark.parametrize("B,K,V,dtype,T", [(12, 6, 4000, torch.float32, 1.0), (40, 7, 20011, torch.bfloat16, 0.8),
                                           (9, 64, 1024, torch.float32, 1.0), (5, 3, 999, torch.float32, 0.7)])
def test_random_lengths_against_oracle(ssv, B, K, V, dtype, T):
    w = synth.gaussian(B, K, V, sigma=2.0, noise=0.6, dtype=dtype, temperature=T, seed=B * 31 + K)
    rng = np.random.default_rng(B + K)
    lengths = rng.integers(0, K + 1, size=B).tolist()
    lengths[0] = 0
    lengths[-1] = K
    off, out = run(ssv, w, lengths, w.temperature)
    assert int(out.status.item()) == 0
    check(w, lengths, w.temperature, off, out)


def test_all_rows_bonus_only(ssv):
    w = synth.gaussian(6, 2, 3000, sigma=2.0, noise=0.5, dtype=torch.float32, temperature=1.0, seed=3)
    lengths = [0] * 6
    off, out = run(ssv, w, lengths, 1.0)
    assert out.n_accepted.cpu().tolist() == [0] * 6
    check(w, lengths, 1.0, off, out)


def test_full_vocab_verify_batch(ssv):
    """The verify batch (B=32, K=4, V=151936) with lengths 0..4 per row."""
    w = synth.entropy_mix(seed=515)
    lengths = [(b * 7) % 5 for b in range(w.shape[0])]
    off, out = run(ssv, w, lengths, 1.0)
    assert int(out.status.item()) == 0
    check(w, lengths, 1.0, off, out)


def test_schedule_then_ragged_verify(ssv):
    """overlap -> prefix survivals -> scheduled lengths -> flattened verify."""
    w = synth.entropy_mix(seed=616)
    B, K, V = w.shape
    o = ssv.overlap(w.target.to(DEV), w.draft.to(DEV), 1.0)
    sps = (2000.0 / (1.0 + np.arange(B * (K + 1) + 1) / 40.0)).astype(np.float32)
    lengths, _ = ssv.schedule_lengths(o.prefix_survival, torch.from_numpy(sps).to(DEV))
    torch.cuda.synchronize()
    lengths = lengths.cpu().tolist()
    assert 0 < sum(lengths) < B * K  # a real trade-off for this table
    off, out = run(ssv, w, lengths, 1.0)
    check(w, lengths, 1.0, off, out)


def test_bad_offsets_and_workspace(ssv):
    w = synth.gaussian(4, 3, 1000, sigma=2.0, noise=0.5, dtype=torch.float32, temperature=1.0, seed=4)
    off, tg, dr, tok, ua = flatten(w, [1, 2, 3, 0])
    units = tg.shape[0]
    ws = torch.zeros(ssv.lib().spec_verify_ragged_workspace_bytes(4, units, 1000), dtype=torch.uint8, device=DEV)
    bad = off.copy()
    bad[2] = bad[1] - 1  # row 1 runs backwards
    out = ssv.verify_ragged(tg.to(DEV), dr.to(DEV), torch.from_numpy(bad).to(DEV), tok.to(DEV), ua.to(DEV),
                            w.u_final.to(DEV), 1.0, workspace=ws)
    torch.cuda.synchronize()
    assert int(out.status.item()) & ssv.DEV_BAD_OFFSETS
    assert int(ws.count_nonzero()) == 0
    good = ssv.verify_ragged(tg.to(DEV), dr.to(DEV), torch.from_numpy(off).to(DEV), tok.to(DEV), ua.to(DEV),
                             w.u_final.to(DEV), 1.0, workspace=ws)
    again = ssv.verify_ragged(tg.to(DEV), dr.to(DEV), torch.from_numpy(off).to(DEV), tok.to(DEV), ua.to(DEV),
                              w.u_final.to(DEV), 1.0, workspace=ws)
    torch.cuda.synchronize()
    assert int(good.status.item()) == 0 and int(ws.count_nonzero()) == 0
    assert torch.equal(good.tokens, again.tokens) and torch.equal(good.alpha, again.alpha)
    check(w, [1, 2, 3, 0], 1.0, off, good)
