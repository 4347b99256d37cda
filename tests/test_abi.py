"""The C-ABI library loads, exports every symbol the header declares, and
rejects bad arguments before touching the GPU (CPU-only tests)."""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def L():
    import sampling_spec_verify_gb300 as ssv
    if not os.path.exists(ssv.LIB_PATH):
        from sampling_spec_verify_gb300 import build
        build.build()
    return ssv.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(spec_[a-z0-9_]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("spec_verify", "spec_overlap", "spec_e2e_tv_fwd_bwd", "spec_status_string",
                 "spec_verify_workspace_bytes", "spec_overlap_workspace_bytes", "spec_e2e_tv_workspace_bytes",
                 "spec_diagnostics", "spec_diagnostics_workspace_bytes", "spec_truncate_logits",
                 "spec_schedule_lengths", "spec_verify_ragged", "spec_verify_ragged_workspace_bytes",
                 "spec_verify_relaxed", "spec_tree_mask", "spec_tree_verify_greedy",
                 "spec_tree_verify_workspace_bytes", "spec_selftest_bounded_wait"):
        assert want in names


def test_library_exports_every_declared_symbol(L):
    import sampling_spec_verify_gb300 as ssv
    out = subprocess.run(["nm", "-D", "--defined-only", ssv.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(L, name)


def test_status_strings_and_version(L):
    assert L.spec_abi_version() == 2
    assert L.spec_status_string(0) == b"ok"
    assert L.spec_status_string(1) == b"invalid argument"
    assert L.spec_status_string(99) == b"unknown status"
    # no kernel is launched without a GPU; the counter answers all the same
    assert L.spec_kernel_launches() == 0


def test_workspace_sizes(L):
    assert L.spec_verify_workspace_bytes(32, 4, 151936) >= 32 * 5 * 16 + 32 * 4
    assert L.spec_verify_workspace_bytes(-1, 4, 10) == 0
    assert L.spec_verify_workspace_bytes(1, 65, 10) == 0
    assert L.spec_e2e_tv_workspace_bytes(256, 7, 151936) >= 256 * 7 * 32
    assert L.spec_overlap_workspace_bytes(8, 4, 100) >= 32
    assert L.spec_diagnostics_workspace_bytes(8, 4, 100) >= 3 * 32 * 16 * 4
    assert L.spec_diagnostics_workspace_bytes(8, 65, 100) == 0


def test_argument_validation_without_gpu(L):
    fake = ctypes.c_void_p(0x1000)
    ws = ctypes.c_void_p(0x2000)
    # bad dims and dtype
    assert L.spec_verify(fake, fake, 1, 2, -1, 10, 1.0, fake, fake, fake, fake, fake, None, None, ws, 1 << 20, None) == 1
    assert L.spec_verify(fake, fake, 7, 2, 2, 10, 1.0, fake, fake, fake, fake, fake, None, None, ws, 1 << 20, None) == 1
    assert L.spec_verify(fake, fake, 1, 2, 2, 0, 1.0, fake, fake, fake, fake, fake, None, None, ws, 1 << 20, None) == 1
    # negative / NaN temperature
    assert L.spec_verify(fake, fake, 1, 2, 2, 10, -1.0, fake, fake, fake, fake, fake, None, None, ws, 1 << 20, None) == 1
    assert L.spec_verify(fake, fake, 1, 2, 2, 10, float("nan"), fake, fake, fake, fake, fake, None, None, ws, 1 << 20,
                         None) == 1
    # empty batch: nothing to do
    assert L.spec_verify(None, None, 1, 0, 2, 10, 1.0, None, None, None, None, None, None, None, None, 0, None) == 0
    # missing outputs, missing draft at T > 0, missing uniforms
    assert L.spec_verify(fake, fake, 1, 2, 2, 10, 1.0, fake, fake, fake, None, fake, None, None, ws, 1 << 20, None) == 1
    assert L.spec_verify(fake, None, 1, 2, 2, 10, 1.0, fake, fake, fake, fake, fake, None, None, ws, 1 << 20, None) == 1
    assert L.spec_verify(fake, fake, 1, 2, 2, 10, 1.0, fake, None, fake, fake, fake, None, None, ws, 1 << 20, None) == 1
    # workspace too small / unaligned
    assert L.spec_verify(fake, fake, 1, 2, 2, 10, 1.0, fake, fake, fake, fake, fake, None, None, ws, 8, None) == 1
    assert L.spec_verify(fake, fake, 1, 2, 2, 10, 1.0, fake, fake, fake, fake, fake, None, None,
                         ctypes.c_void_p(0x2004), 1 << 20, None) == 1
    # E2E needs T > 0 and a loss pointer
    assert L.spec_e2e_tv_fwd_bwd(fake, fake, 1, 2, 2, 2, 10, 0.0, 1.0, fake, None, fake, None, ws, 1 << 20, None) == 1
    assert L.spec_e2e_tv_fwd_bwd(fake, fake, 1, 2, 2, 2, 10, 1.0, 1.0, None, None, fake, None, ws, 1 << 20, None) == 1
    # overlap: KT < K, missing alpha
    assert L.spec_overlap(fake, fake, 1, 2, 3, 2, 10, 1.0, fake, None, None, None, None, ws, 1 << 20, None) == 1
    assert L.spec_overlap(fake, fake, 1, 2, 3, 3, 10, 1.0, None, None, None, None, None, ws, 1 << 20, None) == 1
    # diagnostics: T > 0, KT >= K, workspace large enough; empty batch is a no-op
    assert L.spec_diagnostics(fake, fake, 1, 2, 2, 2, 10, 0.0, fake, None, None, None, None, None, ws, 1 << 20,
                              None) == 1
    assert L.spec_diagnostics(fake, fake, 1, 2, 3, 2, 10, 1.0, fake, None, None, None, None, None, ws, 1 << 20,
                              None) == 1
    assert L.spec_diagnostics(fake, fake, 1, 2, 2, 2, 10, 1.0, fake, None, None, None, None, None, ws, 8, None) == 1
    assert L.spec_diagnostics(None, None, 1, 0, 2, 2, 10, 1.0, None, None, None, None, None, None, None, 0, None) == 0
    # truncation: top_k >= 0, top_p in (0, 1], T > 0 when top-p is on; no rows is a no-op
    assert L.spec_truncate_logits(fake, fake, 1, 2, 10, 1.0, -1, 1.0, None, None) == 1
    assert L.spec_truncate_logits(fake, fake, 1, 2, 10, 1.0, 3, 0.0, None, None) == 1
    assert L.spec_truncate_logits(fake, fake, 1, 2, 10, 1.0, 3, 1.5, None, None) == 1
    assert L.spec_truncate_logits(fake, fake, 1, 2, 10, 0.0, 3, 0.5, None, None) == 1
    assert L.spec_truncate_logits(fake, ctypes.c_void_p(0x1004), 1, 2, 10, 1.0, 3, 1.0, None, None) == 1
    assert L.spec_truncate_logits(None, None, 1, 0, 10, 1.0, 3, 0.5, None, None) == 0
    # scheduling: 1 <= L <= 64, a table covering B = 0 .. R(1 + L), R * L <= 16384
    assert L.spec_schedule_lengths(fake, 2, 0, fake, 100, fake, None, None, None) == 1
    assert L.spec_schedule_lengths(fake, 2, 65, fake, 1000, fake, None, None, None) == 1
    assert L.spec_schedule_lengths(fake, 2, 3, fake, 8, fake, None, None, None) == 1
    assert L.spec_schedule_lengths(fake, 16385, 1, fake, 40000, fake, None, None, None) == 2
    assert L.spec_schedule_lengths(None, 0, 3, None, 0, None, None, None, None) == 0
    # ragged verify: T > 0, B <= units <= 65 B, a large enough workspace; no rows is a no-op
    assert L.spec_verify_ragged(fake, fake, 1, 2, fake, 5, 10, 0.0, fake, fake, fake, fake, fake, None, None, ws,
                                1 << 20, None) == 1
    assert L.spec_verify_ragged(fake, fake, 1, 2, fake, 1, 10, 1.0, fake, fake, fake, fake, fake, None, None, ws,
                                1 << 20, None) == 1
    assert L.spec_verify_ragged(fake, fake, 1, 2, fake, 200, 10, 1.0, fake, fake, fake, fake, fake, None, None, ws,
                                1 << 20, None) == 1
    assert L.spec_verify_ragged(fake, fake, 1, 2, fake, 5, 10, 1.0, fake, fake, fake, fake, fake, None, None, ws,
                                8, None) == 1
    assert L.spec_verify_ragged(None, None, 1, 0, None, 0, 10, 1.0, None, None, None, None, None, None, None, None,
                                0, None) == 0
    assert L.spec_verify_ragged_workspace_bytes(4, 3, 10) == 0
    # relaxed verify: T > 0, delta >= 0; no rows is a no-op
    assert L.spec_verify_relaxed(fake, fake, 1, 2, 2, 10, 0.0, 3, 1.0, fake, fake, fake, fake, None, None, ws,
                                 1 << 20, None) == 1
    assert L.spec_verify_relaxed(fake, fake, 1, 2, 2, 10, 1.0, 3, -1.0, fake, fake, fake, fake, None, None, ws,
                                 1 << 20, None) == 1
    assert L.spec_verify_relaxed(None, None, 1, 0, 2, 10, 1.0, 3, 1.0, None, None, None, None, None, None, None,
                                 0, None) == 0
    # trees: sizes >= 0, a workspace for the argmax of every slot; empty is a no-op
    assert L.spec_tree_mask(fake, -1, 3, fake, None, None, None) == 1
    assert L.spec_tree_mask(None, 0, 3, None, None, None, None) == 0
    assert L.spec_tree_verify_greedy(fake, 1, 2, 3, 10, fake, fake, fake, fake, fake, None, ws, 8, None) == 1
    assert L.spec_tree_verify_greedy(None, 1, 0, 3, 10, None, None, None, None, None, None, None, 0, None) == 0
    assert L.spec_tree_verify_workspace_bytes(2, 3, 10) >= 2 * 4 * 4
    # bounded-wait self-test: a limit in [1 ns, 10 s] and a status word
    assert L.spec_selftest_bounded_wait(0, fake, None) == 1
    assert L.spec_selftest_bounded_wait(10_000_000_001, fake, None) == 1
    assert L.spec_selftest_bounded_wait(1_000_000, None, None) == 1
