"""The allocation-free verify entry point.

spec_verify_noalloc is for callers that cannot allocate device memory when
they run a verify step (under a runtime whose pool owns all device memory, in
a plugin host that only hands out buffers, in a decode loop that cannot take
cudaMalloc's device-wide synchronisation).  It keeps its scratch in a fixed
device array inside the library.  Here it is called through the C ABI and
must give the same results as spec_verify with a caller-provided workspace,
on two calls in a row (the second call reuses the array the first one left
behind), agree with the fp64 oracle, and answer an empty batch as
spec_verify does.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from sampling_spec_verify_gb300 import synth

pytestmark = pytest.mark.gpu

RTOL, ATOL = 1e-4, 1e-6


def _entry(L):
    fn = L.spec_verify_noalloc
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.restype = i32
    fn.argtypes = [vp, vp, i32, i32, i32, i32, f32, vp, vp, vp, vp, vp, vp, vp, vp]
    return fn


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def test_noalloc_matches_workspace_entry_point():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sampling_spec_verify_gb300 as ssv
    L = ssv.lib()
    fn = _entry(L)
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream(dev)
    cases = [synth.gaussian(16, 4, 30000, sigma=2.0, noise=0.6, dtype=torch.bfloat16, temperature=1.0, seed=41),
             synth.gaussian(9, 7, 20011, sigma=2.0, noise=0.5, dtype=torch.float32, temperature=0.7, seed=42)]
    for w in cases:  # two calls in a row on the same scratch array
        B, K, V = w.shape
        t, d = w.target.to(dev), w.draft.to(dev)
        y, ua, uf = w.draft_tokens.to(dev), w.u_accept.to(dev), w.u_final.to(dev)
        ref = ssv.verify(t, d, y, ua, uf, w.temperature)
        tok = torch.full((B, K + 1), -7, dtype=torch.int32, device=dev)
        n = torch.full((B,), -7, dtype=torch.int32, device=dev)
        a = torch.full((B, K), -7.0, dtype=torch.float32, device=dev)
        st = torch.zeros((1,), dtype=torch.int32, device=dev)
        code = 1 if t.dtype == torch.bfloat16 else 0
        rc = fn(_p(t), _p(d), code, B, K, V, w.temperature, _p(y), _p(ua), _p(uf), _p(tok), _p(n), _p(a), _p(st),
                ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0, L.spec_status_string(rc)
        torch.cuda.synchronize()
        assert torch.equal(tok, ref.tokens)
        assert torch.equal(n, ref.n_accepted)
        np.testing.assert_allclose(a.cpu().numpy(), ref.alpha.cpu().numpy(), rtol=RTOL, atol=ATOL)
        assert int(st.item()) == 0
        # and the fp64 oracle, on every row it does not flag as a near tie
        orc = oracle.verify(synth.f64(w.target), synth.f64(w.draft), w.draft_tokens.numpy(), w.u_accept.numpy(),
                            w.u_final.numpy(), w.temperature)
        ok = ~orc.flagged
        assert (tok.cpu().numpy()[ok] == orc.tokens[ok]).all()
        assert (n.cpu().numpy()[ok] == orc.n_accepted[ok]).all()
        np.testing.assert_allclose(a.cpu().numpy(), orc.alpha, rtol=RTOL, atol=ATOL)


def test_noalloc_empty_batch_like_spec_verify():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sampling_spec_verify_gb300 as ssv
    L = ssv.lib()
    fn = _entry(L)
    # B = 0: nothing to do, SPEC_OK, as spec_verify answers (no pointer is touched)
    assert fn(None, None, 1, 0, 4, 1000, 1.0, None, None, None, None, None, None, None, None) == 0
    # invalid dimensions and temperature are rejected like spec_verify rejects them
    assert fn(None, None, 1, 0, 4, 0, 1.0, None, None, None, None, None, None, None, None) == 1
    assert fn(None, None, 1, 0, 4, 1000, -1.0, None, None, None, None, None, None, None, None) == 1
    assert fn(None, None, 1, -1, 4, 1000, 1.0, None, None, None, None, None, None, None, None) == 1


def test_noalloc_rejects_sizes_beyond_its_array():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sampling_spec_verify_gb300 as ssv
    L = ssv.lib()
    fn = _entry(L)
    # 100,000 rows at K = 7 need far more than the fixed scratch array.  Every
    # pointer is null: were the size check ever to let this through,
    # spec_verify's own null checks would answer SPEC_ERR_INVALID_ARG before
    # any launch.
    rc = fn(None, None, 1, 100000, 7, 1024, 1.0, None, None, None, None, None, None, None, None)
    assert rc == 2  # SPEC_ERR_UNSUPPORTED
