"""Failure detection without a GPU fault.

A bounded wait that runs out is reported on the device status word, the
kernel returns normally, and the context stays usable.  The wait is the one
the sweep uses on its bulk copies.  Here it runs on an mbarrier that nothing
completes, with no copy in flight.
"""

import time

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


def _small_verify_matches_oracle(ssv):
    g = torch.Generator().manual_seed(9)
    B, K, V = 3, 2, 257
    zt = torch.randn(B, K + 1, V, generator=g)
    zd = (zt[:, :K] + 0.5 * torch.randn(B, K, V, generator=g)).contiguous()
    y = torch.randint(0, V, (B, K), generator=g, dtype=torch.int32)
    ua = torch.rand(B, K, generator=g)
    uf = torch.rand(B, generator=g)
    out = ssv.verify(zt.to(DEV), zd.to(DEV), y.to(DEV), ua.to(DEV), uf.to(DEV), 1.0)
    torch.cuda.synchronize()
    assert int(out.status.item()) == 0
    ref = oracle.verify(synth.f64(zt), synth.f64(zd), y.numpy(), ua.numpy(), uf.numpy(), 1.0)
    ok = ~ref.flagged
    assert ((out.tokens.cpu().numpy() == ref.tokens).all(axis=1) | ~ok).all()
    assert ((out.n_accepted.cpu().numpy() == ref.n_accepted) | ~ok).all()


def test_wait_that_runs_out_is_reported_and_the_context_survives(ssv):
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ssv.selftest_bounded_wait(2_000_000, status=st)  # 2 ms
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(st.item()) == ssv.DEV_TIMEOUT
    assert dt >= 2e-3, f"the wait gave up after {dt * 1e3:.3f} ms"
    _small_verify_matches_oracle(ssv)


def test_timeout_bit_is_or_ed_into_the_status_word(ssv):
    st = torch.full((1,), ssv.DEV_BAD_TOKEN, dtype=torch.int32, device=DEV)
    ssv.selftest_bounded_wait(1000, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == ssv.DEV_BAD_TOKEN | ssv.DEV_TIMEOUT
    # on a side stream, after the status word's zero fill on the current stream
    s = torch.cuda.Stream()
    st2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ssv.selftest_bounded_wait(100_000, status=st2, stream=s)
    s.synchronize()
    assert int(st2.item()) == ssv.DEV_TIMEOUT
    _small_verify_matches_oracle(ssv)


def test_invalid_limits_are_refused(ssv):
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    for bad in (0, 10_000_000_001):
        with pytest.raises(ssv.SpecError):
            ssv.selftest_bounded_wait(bad, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
