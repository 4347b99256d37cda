"""GPU parity of the candidate-tree kernels against the oracle: the tree
attention mask and depth bit-exact; the greedy tree verify's path, tokens and
accepted counts bit-exact (argmax with the smallest index on ties on both
sides, on the same stored logits)."""

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


def random_parents(rng, B, N):
    par = np.full((B, N), -1, dtype=np.int32)
    for b in range(B):
        for i in range(1, N):
            par[b, i] = int(rng.integers(-1, i))
    return par


def tree_case(rng, B, N, V, dtype, scale=2.0):
    z = torch.from_numpy(rng.normal(size=(B, N + 1, V)).astype(np.float32) * scale)
    z = torch.round(z * 4) / 4  # ties
    z = z.to(dtype)
    par = random_parents(rng, B, N)
    zf = synth.f64(z)
    tok = np.zeros((B, N), dtype=np.int32)
    for b in range(B):
        for i in range(N):
            if rng.uniform() < 0.6:  # the parent slot's argmax: the walk can go deep
                tok[b, i] = oracle.argmax_first(zf[b, par[b, i] + 1])
            else:
                tok[b, i] = int(rng.integers(0, V))
    return z, par, tok


def test_mask_against_oracle(ssv):
    rng = np.random.default_rng(51)
    for B, N in ((1, 1), (3, 7), (2, 64), (4, 200)):
        par = random_parents(rng, B, N)
        par[0, : min(N, 5)] = np.arange(-1, min(N, 5) - 1)  # a chain start
        mask, depth = ssv.tree_mask(torch.from_numpy(par).to(DEV))
        torch.cuda.synchronize()
        m, d = mask.cpu().numpy().astype(bool), depth.cpu().numpy()
        for b in range(B):
            M, D = oracle.tree_mask(par[b])
            assert (m[b] == M).all() and (d[b] == D).all()


@pytest.mark.parametrize("B,N,V,dtype", [(6, 9, 3000, torch.float32), (5, 33, 20011, torch.bfloat16),
                                         (8, 16, 151936, torch.bfloat16), (3, 64, 999, torch.float32)])
def test_greedy_against_oracle(ssv, B, N, V, dtype):
    rng = np.random.default_rng(B * 100 + N)
    z, par, tok = tree_case(rng, B, N, V, dtype)
    out = ssv.tree_verify_greedy(z.to(DEV), torch.from_numpy(par).to(DEV), torch.from_numpy(tok).to(DEV))
    torch.cuda.synchronize()
    ref = oracle.tree_verify_greedy(synth.f64(z), par, tok)
    assert int(out.status.item()) == 0
    assert out.n_accepted.cpu().numpy().tolist() == ref.n_accepted.tolist()
    assert out.path.cpu().numpy().tolist() == ref.path.tolist()
    assert out.tokens.cpu().numpy().tolist() == ref.tokens.tolist()
    assert ref.n_accepted.max() >= 2  # the case exercises depth


def test_chain_tree_equals_linear_greedy(ssv):
    w = synth.gaussian(6, 5, 4096, sigma=2.0, noise=0.3, dtype=torch.bfloat16, temperature=0.0, seed=61)
    B, K, V = w.shape
    lin = ssv.verify(w.target.to(DEV), None, w.draft_tokens.to(DEV), None, None, 0.0)
    par = torch.arange(-1, K - 1, dtype=torch.int32).repeat(B, 1)
    tr = ssv.tree_verify_greedy(w.target.to(DEV), par.to(DEV), w.draft_tokens.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(tr.n_accepted, lin.n_accepted)
    assert torch.equal(tr.tokens, lin.tokens)


def test_bad_parent_map(ssv):
    rng = np.random.default_rng(7)
    z, par, tok = tree_case(rng, 2, 4, 512, torch.float32)
    par[1, 2] = 3  # a parent after its child
    out = ssv.tree_verify_greedy(z.to(DEV), torch.from_numpy(par).to(DEV), torch.from_numpy(tok).to(DEV))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ssv.tree_mask(torch.from_numpy(par).to(DEV), status=st)
    torch.cuda.synchronize()
    assert int(out.status.item()) & ssv.DEV_BAD_OFFSETS and int(st.item()) & ssv.DEV_BAD_OFFSETS
    n = out.n_accepted.cpu().tolist()
    assert n[1] == -1 and n[0] == oracle.tree_verify_greedy(synth.f64(z[:1]), par[:1], tok[:1]).n_accepted[0]
