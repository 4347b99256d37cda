"""Speculative-sampling verify on GB300: Python binding of the C ABI.

The functions here only marshal arguments: every step of the verify, overlap
and E2E-TV computations runs in the CUDA kernels of ``libspec_verify.so``.
PyTorch provides device memory and streams.  There is no CPU fallback: if the
library is missing, every call raises.

Entry points (same names as the C ABI, see include/spec_verify.h):

* ``verify``          -- batched draft/verify step (acceptance, residual
                         correction, bonus token, greedy at T == 0);
* ``verify_ragged``   -- the same with a length of its own per row, over
                         flattened tensors and row offsets;
* ``verify_relaxed``  -- LOSSY relaxed acceptance (target top-k rank and
                         log-probability gap);
* ``tree_mask``, ``tree_verify_greedy`` -- candidate trees: the attention
                         mask of a parent map, and the greedy verify that
                         commits one path;
* ``overlap``         -- alpha = sum min(p, q), TV, prefix survival, E[tau];
* ``e2e_tv_fwd_bwd``  -- E2E-TV loss and its draft-logit gradient;
* ``diagnostics``     -- alpha, target entropy, cross-entropy, KL and the
                         target-only acceptance p(argmax q) per position;
* ``truncate_logits`` -- top-k / top-p truncation, to apply identically to
                         target and draft logits before ``verify``;
* ``schedule_lengths`` -- verify lengths maximising tau * SPS(B) over prefix
                         survivals and a throughput table.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

__all__ = [
    "SpecError", "lib", "verify", "verify_ragged", "verify_relaxed", "tree_mask", "tree_verify_greedy", "overlap", "e2e_tv_fwd_bwd", "diagnostics", "truncate_logits", "schedule_lengths", "selftest_bounded_wait", "launch_shape", "kernel_launches", "set_kernel_override",
    "set_launch_override", "VerifyOutput", "OverlapOutput", "E2EOutput", "DiagOutput", "TreeOutput", "HostVerifier",
    "DEV_BAD_TOKEN", "DEV_BAD_LOGITS", "DEV_BAD_UNIFORM", "DEV_TIMEOUT", "DEV_EMPTY_RESIDUAL", "DEV_BAD_OFFSETS",
    "SPEC_OK", "SPEC_ERR_INVALID_ARG", "SPEC_ERR_UNSUPPORTED", "SPEC_ERR_CUDA",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libspec_verify.so")

SPEC_OK, SPEC_ERR_INVALID_ARG, SPEC_ERR_UNSUPPORTED, SPEC_ERR_CUDA = 0, 1, 2, 3
SPEC_F32, SPEC_BF16 = 0, 1
DEV_BAD_TOKEN, DEV_BAD_LOGITS, DEV_BAD_UNIFORM, DEV_TIMEOUT, DEV_EMPTY_RESIDUAL = 1, 2, 4, 8, 16
DEV_BAD_OFFSETS = 32

_lib = None


class SpecError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        msg = lib().spec_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{what}: {msg} (status {status})")


def lib():
    """The loaded C library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` "
            "(or sampling_spec_verify_gb300.build.build())")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.spec_abi_version.restype = i32
    L.spec_kernel_launches.restype = ctypes.c_ulonglong
    L.spec_kernel_launches.argtypes = []
    L.spec_status_string.restype = ctypes.c_char_p
    L.spec_status_string.argtypes = [i32]
    L.spec_verify_workspace_bytes.restype = sz
    L.spec_verify_workspace_bytes.argtypes = [i32, i32, i32]
    L.spec_verify.restype = i32
    L.spec_verify.argtypes = [vp, vp, i32, i32, i32, i32, f32, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.spec_overlap_workspace_bytes.restype = sz
    L.spec_overlap_workspace_bytes.argtypes = [i32, i32, i32]
    L.spec_overlap.restype = i32
    L.spec_overlap.argtypes = [vp, vp, i32, i32, i32, i32, i32, f32, vp, vp, vp, vp, vp, vp, sz, vp]
    L.spec_e2e_tv_workspace_bytes.restype = sz
    L.spec_e2e_tv_workspace_bytes.argtypes = [i32, i32, i32]
    L.spec_e2e_tv_fwd_bwd.restype = i32
    L.spec_e2e_tv_fwd_bwd.argtypes = [vp, vp, i32, i32, i32, i32, i32, f32, f32, vp, vp, vp, vp, vp, sz, vp]
    L.spec_diagnostics_workspace_bytes.restype = sz
    L.spec_diagnostics_workspace_bytes.argtypes = [i32, i32, i32]
    L.spec_diagnostics.restype = i32
    L.spec_diagnostics.argtypes = [vp, vp, i32, i32, i32, i32, i32, f32, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.spec_truncate_logits.restype = i32
    L.spec_truncate_logits.argtypes = [vp, vp, i32, i32, i32, f32, i32, f32, vp, vp]
    L.spec_schedule_lengths.restype = i32
    L.spec_schedule_lengths.argtypes = [vp, i32, i32, vp, i32, vp, vp, vp, vp]
    L.spec_verify_ragged_workspace_bytes.restype = sz
    L.spec_verify_ragged_workspace_bytes.argtypes = [i32, i32, i32]
    L.spec_verify_ragged.restype = i32
    L.spec_verify_ragged.argtypes = [vp, vp, i32, i32, vp, i32, i32, f32, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.spec_verify_relaxed.restype = i32
    L.spec_verify_relaxed.argtypes = [vp, vp, i32, i32, i32, i32, f32, i32, f32, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.spec_tree_mask.restype = i32
    L.spec_tree_mask.argtypes = [vp, i32, i32, vp, vp, vp, vp]
    L.spec_tree_verify_workspace_bytes.restype = sz
    L.spec_tree_verify_workspace_bytes.argtypes = [i32, i32, i32]
    L.spec_tree_verify_greedy.restype = i32
    L.spec_tree_verify_greedy.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.spec_selftest_bounded_wait.restype = i32
    L.spec_selftest_bounded_wait.argtypes = [ctypes.c_uint64, vp, vp]
    L.spec_launch_shape.restype = i32
    L.spec_launch_shape.argtypes = [i32, i32, i32] + [ctypes.POINTER(i32)] * 5
    L.spec_set_launch_override.restype = None
    L.spec_set_launch_override.argtypes = [i32, i32]
    L.spec_set_kernel_override.restype = None
    L.spec_set_kernel_override.argtypes = [i32]
    _lib = L
    return L


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    if t.dtype == torch.float32:
        return SPEC_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _need(t: torch.Tensor, name: str, dtype=None, shape=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}")


def _stream_handle(stream: Optional[torch.cuda.Stream], device):
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream), s


_WS = {}


def _workspace(nbytes: int, device, stream) -> torch.Tensor:
    """A zero-filled workspace cached per (device, stream).  The library
    leaves it zero-filled after every completed call."""
    key = (device.index, stream.cuda_stream)
    ws = _WS.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
        _WS[key] = ws
    return ws


def _check(status: int, what: str):
    if status != SPEC_OK:
        raise SpecError(status, what)


def kernel_launches() -> int:
    """Kernels the library has launched in this process (host-side count)."""
    return int(lib().spec_kernel_launches())


def set_kernel_override(kernel: int = 0) -> None:
    """Sweep kernel of later calls: 0 automatic, 1 the single-read sweep,
    2 the two-pass sweep where it applies."""
    lib().spec_set_kernel_override(int(kernel))


def set_launch_override(cluster_ctas: int = 0, stages: int = 0) -> None:
    """Force the CTAs per cluster (1..16) and shared-memory stages (1 or 2)
    of later launches; 0 = automatic."""
    lib().spec_set_launch_override(int(cluster_ctas), int(stages))


def launch_shape(dtype: torch.dtype, units: int, V: int):
    """(cluster CTAs, threads per CTA, dynamic shared bytes, clusters, stages)
    of a verify sweep over `units` (row, position) pairs."""
    v = [ctypes.c_int() for _ in range(5)]
    code = SPEC_BF16 if dtype == torch.bfloat16 else SPEC_F32
    _check(lib().spec_launch_shape(code, units, V, *[ctypes.byref(x) for x in v]), "spec_launch_shape")
    return tuple(x.value for x in v)


# ---------------------------------------------------------------------------
# verify
# ---------------------------------------------------------------------------

@dataclass
class VerifyOutput:
    tokens: torch.Tensor       # int32 [B, K+1]
    n_accepted: torch.Tensor   # int32 [B]
    alpha: Optional[torch.Tensor]  # float32 [B, K]
    status: torch.Tensor       # int32 [1] device status word


def verify(target: torch.Tensor, draft: Optional[torch.Tensor], draft_tokens: torch.Tensor,
           u_accept: Optional[torch.Tensor], u_final: Optional[torch.Tensor], temperature: float, *,
           want_alpha: bool = True, out: Optional[VerifyOutput] = None,
           workspace: Optional[torch.Tensor] = None,
           stream: Optional[torch.cuda.Stream] = None) -> VerifyOutput:
    """Batched verify of K drafted tokens per row (see spec_verify in the C
    header).  target [B, K+1, V], draft [B, K, V] (bf16 or fp32),
    draft_tokens int32 [B, K], u_accept float32 [B, K], u_final float32 [B]."""
    L = lib()
    _need(target, "target")
    B, K1, V = target.shape
    K = K1 - 1
    dev = target.device
    greedy = float(temperature) == 0.0
    if draft is not None:
        _need(draft, "draft", dtype=target.dtype, shape=(B, K, V), device=dev)
    _need(draft_tokens, "draft_tokens", dtype=torch.int32, shape=(B, K), device=dev)
    if not greedy:
        _need(u_accept, "u_accept", dtype=torch.float32, shape=(B, K), device=dev)
        _need(u_final, "u_final", dtype=torch.float32, shape=(B,), device=dev)
    want_alpha = want_alpha and draft is not None
    if out is None:
        out = VerifyOutput(
            torch.empty((B, K + 1), dtype=torch.int32, device=dev),
            torch.empty((B,), dtype=torch.int32, device=dev),
            torch.empty((B, K), dtype=torch.float32, device=dev) if want_alpha else None,
            torch.zeros((1,), dtype=torch.int32, device=dev))
    sh, s = _stream_handle(stream, dev)
    need = L.spec_verify_workspace_bytes(B, K, V)
    ws = workspace if workspace is not None else _workspace(need, dev, s)
    st = L.spec_verify(_ptr(target), _ptr(draft), _dtype_code(target), B, K, V, float(temperature),
                       _ptr(draft_tokens), _ptr(u_accept), _ptr(u_final), _ptr(out.tokens),
                       _ptr(out.n_accepted), _ptr(out.alpha), _ptr(out.status), _ptr(ws),
                       ws.numel() * ws.element_size(), sh)
    _check(st, "spec_verify")
    return out


def verify_ragged(target: torch.Tensor, draft: Optional[torch.Tensor], row_offsets: torch.Tensor,
                  draft_tokens: Optional[torch.Tensor], u_accept: Optional[torch.Tensor], u_final: torch.Tensor,
                  temperature: float, *, want_alpha: bool = True, workspace: Optional[torch.Tensor] = None,
                  stream: Optional[torch.cuda.Stream] = None) -> VerifyOutput:
    """Verify with a length of its own per row (see spec_verify_ragged in
    the C header).  target [units, V]: row r's drafted positions then its
    bonus position at rows row_offsets[r] .. row_offsets[r+1]-1; draft
    [units - B, V], draft_tokens and u_accept [units - B] in the same
    flattened order; row_offsets int32 [B + 1]; u_final [B].  Returns tokens
    [units] (flattened like target), n_accepted [B], alpha [units - B]."""
    L = lib()
    _need(target, "target")
    units, V = target.shape
    dev = target.device
    _need(row_offsets, "row_offsets", dtype=torch.int32, device=dev)
    B = row_offsets.numel() - 1
    nd = units - B
    _need(u_final, "u_final", dtype=torch.float32, shape=(B,), device=dev)
    if nd > 0:
        _need(draft, "draft", dtype=target.dtype, shape=(nd, V), device=dev)
        _need(draft_tokens, "draft_tokens", dtype=torch.int32, shape=(nd,), device=dev)
        _need(u_accept, "u_accept", dtype=torch.float32, shape=(nd,), device=dev)
    out = VerifyOutput(torch.empty((units,), dtype=torch.int32, device=dev),
                       torch.empty((B,), dtype=torch.int32, device=dev),
                       torch.empty((nd,), dtype=torch.float32, device=dev) if want_alpha and nd > 0 else None,
                       torch.zeros((1,), dtype=torch.int32, device=dev))
    sh, s = _stream_handle(stream, dev)
    need = L.spec_verify_ragged_workspace_bytes(B, units, V)
    ws = workspace if workspace is not None else _workspace(need, dev, s)
    st = L.spec_verify_ragged(_ptr(target), _ptr(draft), _dtype_code(target), B, _ptr(row_offsets), units, V,
                              float(temperature), _ptr(draft_tokens), _ptr(u_accept), _ptr(u_final),
                              _ptr(out.tokens), _ptr(out.n_accepted), _ptr(out.alpha), _ptr(out.status), _ptr(ws),
                              ws.numel() * ws.element_size(), sh)
    _check(st, "spec_verify_ragged")
    return out


def verify_relaxed(target: torch.Tensor, draft: torch.Tensor, draft_tokens: torch.Tensor, u_final: torch.Tensor,
                   temperature: float, top_k: int = 0, delta: float = float("inf"), *, want_alpha: bool = True,
                   workspace: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None) -> VerifyOutput:
    """LOSSY verify: a draft is accepted while it ranks in the target's
    top_k (0: no rank condition) and its log-probability lies within delta
    of the target's largest (inf: no gap condition); the first rejection
    draws from the full target.  Shapes as ``verify``, without u_accept."""
    L = lib()
    _need(target, "target")
    B, K1, V = target.shape
    K = K1 - 1
    dev = target.device
    _need(draft, "draft", dtype=target.dtype, shape=(B, K, V), device=dev)
    _need(draft_tokens, "draft_tokens", dtype=torch.int32, shape=(B, K), device=dev)
    _need(u_final, "u_final", dtype=torch.float32, shape=(B,), device=dev)
    if K == 0:
        draft = draft_tokens = None  # an empty tensor may have no storage
    out = VerifyOutput(torch.empty((B, K + 1), dtype=torch.int32, device=dev),
                       torch.empty((B,), dtype=torch.int32, device=dev),
                       torch.empty((B, K), dtype=torch.float32, device=dev) if want_alpha else None,
                       torch.zeros((1,), dtype=torch.int32, device=dev))
    sh, s = _stream_handle(stream, dev)
    need = L.spec_verify_workspace_bytes(B, K, V)
    ws = workspace if workspace is not None else _workspace(need, dev, s)
    st = L.spec_verify_relaxed(_ptr(target), _ptr(draft), _dtype_code(target), B, K, V, float(temperature),
                               int(top_k), float(delta), _ptr(draft_tokens), _ptr(u_final), _ptr(out.tokens),
                               _ptr(out.n_accepted), _ptr(out.alpha), _ptr(out.status), _ptr(ws),
                               ws.numel() * ws.element_size(), sh)
    _check(st, "spec_verify_relaxed")
    return out


def tree_mask(parent: torch.Tensor, *, status: Optional[torch.Tensor] = None,
              stream: Optional[torch.cuda.Stream] = None):
    """Tree attention mask of parent maps [B, N] (int32, parent[i] < i, -1
    on the prefix): (mask uint8 [B, N, N], depth int32 [B, N])."""
    L = lib()
    _need(parent, "parent", dtype=torch.int32)
    B, N = parent.shape
    dev = parent.device
    mask = torch.empty((B, N, N), dtype=torch.uint8, device=dev)
    depth = torch.empty((B, N), dtype=torch.int32, device=dev)
    sh, _ = _stream_handle(stream, dev)
    _check(L.spec_tree_mask(_ptr(parent), B, N, _ptr(mask), _ptr(depth), _ptr(status), sh), "spec_tree_mask")
    return mask, depth


@dataclass
class TreeOutput:
    path: torch.Tensor        # int32 [B, N]
    tokens: torch.Tensor      # int32 [B, N + 1]
    n_accepted: torch.Tensor  # int32 [B]
    status: torch.Tensor


def tree_verify_greedy(target: torch.Tensor, parent: torch.Tensor, node_tokens: torch.Tensor, *,
                       workspace: Optional[torch.Tensor] = None,
                       stream: Optional[torch.cuda.Stream] = None) -> TreeOutput:
    """Greedy verify of candidate trees: target [B, N + 1, V] (slot 0 after
    the prefix, slot i + 1 after node i), parent and node_tokens [B, N]."""
    L = lib()
    _need(target, "target")
    B, N1, V = target.shape
    N = N1 - 1
    dev = target.device
    _need(parent, "parent", dtype=torch.int32, shape=(B, N), device=dev)
    _need(node_tokens, "node_tokens", dtype=torch.int32, shape=(B, N), device=dev)
    out = TreeOutput(torch.empty((B, N), dtype=torch.int32, device=dev),
                     torch.empty((B, N + 1), dtype=torch.int32, device=dev),
                     torch.empty((B,), dtype=torch.int32, device=dev),
                     torch.zeros((1,), dtype=torch.int32, device=dev))
    sh, s = _stream_handle(stream, dev)
    need = L.spec_tree_verify_workspace_bytes(B, N, V)
    ws = workspace if workspace is not None else _workspace(need, dev, s)
    st = L.spec_tree_verify_greedy(_ptr(target), _dtype_code(target), B, N, V, _ptr(parent), _ptr(node_tokens),
                                   _ptr(out.path), _ptr(out.tokens), _ptr(out.n_accepted), _ptr(out.status),
                                   _ptr(ws), ws.numel() * ws.element_size(), sh)
    _check(st, "spec_tree_verify_greedy")
    return out


# ---------------------------------------------------------------------------
# overlap
# ---------------------------------------------------------------------------

@dataclass
class OverlapOutput:
    alpha: torch.Tensor
    tv: Optional[torch.Tensor]
    prefix_survival: Optional[torch.Tensor]
    expected_accepted: Optional[torch.Tensor]
    status: torch.Tensor


def overlap(target: torch.Tensor, draft: torch.Tensor, temperature: float, *, K: Optional[int] = None,
            want_tv: bool = True, want_survival: bool = True, out: Optional[OverlapOutput] = None,
            workspace: Optional[torch.Tensor] = None,
            stream: Optional[torch.cuda.Stream] = None) -> OverlapOutput:
    """Per-position overlap statistics.  target [B, KT, V] with KT >= K (the
    first K positions are used), draft [B, K, V]."""
    L = lib()
    _need(target, "target")
    _need(draft, "draft", dtype=target.dtype)
    B, KT, V = target.shape
    K = draft.shape[1] if K is None else K
    if tuple(draft.shape) != (B, K, V) or KT < K:
        raise ValueError("draft must be [B, K, V] with K <= target.shape[1]")
    dev = target.device
    if out is None:
        f = lambda *shape: torch.empty(shape, dtype=torch.float32, device=dev)  # noqa: E731
        out = OverlapOutput(f(B, K), f(B, K) if want_tv else None, f(B, K) if want_survival else None,
                            f(B) if want_survival else None, torch.zeros((1,), dtype=torch.int32, device=dev))
    sh, s = _stream_handle(stream, dev)
    need = L.spec_overlap_workspace_bytes(B, K, V)
    ws = workspace if workspace is not None else _workspace(need, dev, s)
    st = L.spec_overlap(_ptr(target), _ptr(draft), _dtype_code(target), B, K, KT, V, float(temperature),
                        _ptr(out.alpha), _ptr(out.tv), _ptr(out.prefix_survival),
                        _ptr(out.expected_accepted), _ptr(out.status), _ptr(ws),
                        ws.numel() * ws.element_size(), sh)
    _check(st, "spec_overlap")
    return out


# ---------------------------------------------------------------------------
# E2E-TV
# ---------------------------------------------------------------------------

@dataclass
class E2EOutput:
    loss: torch.Tensor            # float32 [1]
    alpha: Optional[torch.Tensor]  # float32 [B, K]
    grad: torch.Tensor            # float32 [B, K, V]
    status: torch.Tensor


def e2e_tv_fwd_bwd(target: torch.Tensor, draft: torch.Tensor, temperature: float, grad_scale: float = 1.0, *,
                   K: Optional[int] = None, want_alpha: bool = True, out: Optional[E2EOutput] = None,
                   workspace: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None) -> E2EOutput:
    """E2E-TV loss mean_b sum_j prod_{k<=j} alpha_{b,k} and grad_scale times
    its gradient with respect to the draft logits (target held constant)."""
    L = lib()
    _need(target, "target")
    _need(draft, "draft", dtype=target.dtype)
    B, KT, V = target.shape
    K = draft.shape[1] if K is None else K
    if tuple(draft.shape) != (B, K, V) or KT < K:
        raise ValueError("draft must be [B, K, V] with K <= target.shape[1]")
    dev = target.device
    if out is None:
        out = E2EOutput(torch.empty((1,), dtype=torch.float32, device=dev),
                        torch.empty((B, K), dtype=torch.float32, device=dev) if want_alpha else None,
                        torch.empty((B, K, V), dtype=torch.float32, device=dev),
                        torch.zeros((1,), dtype=torch.int32, device=dev))
    sh, s = _stream_handle(stream, dev)
    need = L.spec_e2e_tv_workspace_bytes(B, K, V)
    ws = workspace if workspace is not None else _workspace(need, dev, s)
    st = L.spec_e2e_tv_fwd_bwd(_ptr(target), _ptr(draft), _dtype_code(target), B, K, KT, V, float(temperature),
                               float(grad_scale), _ptr(out.loss), _ptr(out.alpha), _ptr(out.grad),
                               _ptr(out.status), _ptr(ws), ws.numel() * ws.element_size(), sh)
    _check(st, "spec_e2e_tv_fwd_bwd")
    return out


# ---------------------------------------------------------------------------
# diagnostics
# ---------------------------------------------------------------------------

@dataclass
class DiagOutput:
    alpha: Optional[torch.Tensor]              # float32 [B, K]: sum_v min(p, q)
    entropy: Optional[torch.Tensor]            # H(p), nats
    cross_entropy: Optional[torch.Tensor]      # -sum_v p log q
    kl: Optional[torch.Tensor]                 # KL(p || q)
    alpha_target_only: Optional[torch.Tensor]  # p(argmax q)
    status: torch.Tensor


def diagnostics(target: torch.Tensor, draft: torch.Tensor, temperature: float, *, K: Optional[int] = None,
                out: Optional[DiagOutput] = None, workspace: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None) -> DiagOutput:
    """Per-position alpha, entropy of p, cross-entropy and KL of q against p,
    and the acceptance p(argmax q) of a point-mass drafter, p and q at
    temperature T > 0.  target [B, KT, V] with KT >= K, draft [B, K, V].
    Fields of ``out`` left as None are not computed."""
    L = lib()
    _need(target, "target")
    _need(draft, "draft", dtype=target.dtype)
    B, KT, V = target.shape
    K = draft.shape[1] if K is None else K
    if tuple(draft.shape) != (B, K, V) or KT < K:
        raise ValueError("draft must be [B, K, V] with K <= target.shape[1]")
    dev = target.device
    if out is None:
        f = lambda: torch.empty((B, K), dtype=torch.float32, device=dev)  # noqa: E731
        out = DiagOutput(f(), f(), f(), f(), f(), torch.zeros((1,), dtype=torch.int32, device=dev))
    sh, s = _stream_handle(stream, dev)
    need = L.spec_diagnostics_workspace_bytes(B, K, V)
    ws = workspace if workspace is not None else _workspace(need, dev, s)
    st = L.spec_diagnostics(_ptr(target), _ptr(draft), _dtype_code(target), B, K, KT, V, float(temperature),
                            _ptr(out.alpha), _ptr(out.entropy), _ptr(out.cross_entropy), _ptr(out.kl),
                            _ptr(out.alpha_target_only), _ptr(out.status), _ptr(ws),
                            ws.numel() * ws.element_size(), sh)
    _check(st, "spec_diagnostics")
    return out


# ---------------------------------------------------------------------------
# top-k / top-p truncation
# ---------------------------------------------------------------------------

def truncate_logits(logits: torch.Tensor, temperature: float, top_k: int = 0, top_p: float = 1.0, *,
                    out: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                    stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Top-k then top-p truncation of every row of ``logits`` [..., V]
    (dropped logits become -inf).  Apply it with the same arguments to the
    target and the draft logits of a verify step.  ``out`` may be ``logits``
    (in place); ``status`` is an optional int32 [1] device word."""
    L = lib()
    _need(logits, "logits")
    V = logits.shape[-1]
    rows = logits.numel() // V if V else 0
    if out is None:
        out = torch.empty_like(logits)
    elif out.shape != logits.shape or out.dtype != logits.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor of the shape and dtype of logits")
    sh, _ = _stream_handle(stream, logits.device)
    st = L.spec_truncate_logits(_ptr(logits), _ptr(out), _dtype_code(logits), rows, V, float(temperature),
                                int(top_k), float(top_p), _ptr(status), sh)
    _check(st, "spec_truncate_logits")
    return out


# ---------------------------------------------------------------------------
# verify-length scheduling
# ---------------------------------------------------------------------------

def schedule_lengths(survival: torch.Tensor, sps: torch.Tensor, *, status: Optional[torch.Tensor] = None,
                     stream: Optional[torch.cuda.Stream] = None):
    """Verify lengths l_r maximising tau * SPS(B) for prefix survivals
    ``survival`` [R, L] (float32, e.g. ``overlap(...).prefix_survival``) and
    a throughput table ``sps`` [>= R * (1 + L) + 1] (float32, SPS(B) at index
    B).  Returns (lengths int32 [R], objective float32 [2] = {Theta, tau})."""
    L_ = lib()
    _need(survival, "survival", dtype=torch.float32)
    _need(sps, "sps", dtype=torch.float32, device=survival.device)
    R, L = survival.shape
    dev = survival.device
    lengths = torch.empty((R,), dtype=torch.int32, device=dev)
    objective = torch.empty((2,), dtype=torch.float32, device=dev)
    sh, _ = _stream_handle(stream, dev)
    st = L_.spec_schedule_lengths(_ptr(survival), R, L, _ptr(sps), sps.numel(), _ptr(lengths), _ptr(objective),
                                  _ptr(status), sh)
    _check(st, "spec_schedule_lengths")
    return lengths, objective


# ---------------------------------------------------------------------------
# host-buffer convenience: one verify step from pinned host memory
# ---------------------------------------------------------------------------

def selftest_bounded_wait(limit_ns: int = 2_000_000, *, status: Optional[torch.Tensor] = None,
                          device="cuda", stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Failure-path self-test of the library's bounded wait (see
    spec_selftest_bounded_wait in the C header): one warp waits on an
    mbarrier that nothing completes and gives up after ``limit_ns``.  Returns
    the int32 status word, which holds DEV_TIMEOUT once the stream has run the
    test."""
    L = lib()
    if status is None:
        status = torch.zeros((1,), dtype=torch.int32, device=torch.device(device))
    _need(status, "status", dtype=torch.int32, shape=(1,))
    sh, _ = _stream_handle(stream, status.device)
    _check(L.spec_selftest_bounded_wait(int(limit_ns), _ptr(status), sh), "spec_selftest_bounded_wait")
    return status


class HostVerifier:
    """Runs verify steps whose inputs and outputs live in (pinned) host
    memory: each ``run`` copies the step's inputs to the device, launches the
    verify kernel and copies tokens, accepted counts and overlaps back, all on
    one stream, then waits for the stream."""

    def __init__(self, B: int, K: int, V: int, dtype=torch.bfloat16, device="cuda",
                 stream: Optional[torch.cuda.Stream] = None):
        self.device = torch.device(device)
        self.stream = stream or torch.cuda.Stream(self.device)
        d = self.device
        self.target = torch.empty((B, K + 1, V), dtype=dtype, device=d)
        self.draft = torch.empty((B, K, V), dtype=dtype, device=d)
        self.tokens_in = torch.empty((B, K), dtype=torch.int32, device=d)
        self.ua = torch.empty((B, K), dtype=torch.float32, device=d)
        self.uf = torch.empty((B,), dtype=torch.float32, device=d)
        self.out = VerifyOutput(torch.empty((B, K + 1), dtype=torch.int32, device=d),
                                torch.empty((B,), dtype=torch.int32, device=d),
                                torch.empty((B, K), dtype=torch.float32, device=d),
                                torch.zeros((1,), dtype=torch.int32, device=d))
        self.ws = torch.zeros(max(lib().spec_verify_workspace_bytes(B, K, V), 256), dtype=torch.uint8, device=d)
        self.h2d_bytes = sum(t.numel() * t.element_size()
                             for t in (self.target, self.draft, self.tokens_in, self.ua, self.uf))
        self.d2h_bytes = sum(t.numel() * t.element_size() for t in (self.out.tokens, self.out.n_accepted,
                                                                   self.out.alpha))

    def run(self, target_h, draft_h, tokens_h, ua_h, uf_h, temperature, tokens_out_h, n_acc_out_h, alpha_out_h):
        with torch.cuda.stream(self.stream):
            self.target.copy_(target_h, non_blocking=True)
            self.draft.copy_(draft_h, non_blocking=True)
            self.tokens_in.copy_(tokens_h, non_blocking=True)
            self.ua.copy_(ua_h, non_blocking=True)
            self.uf.copy_(uf_h, non_blocking=True)
            verify(self.target, self.draft, self.tokens_in, self.ua, self.uf, temperature,
                   out=self.out, workspace=self.ws, stream=self.stream)
            tokens_out_h.copy_(self.out.tokens, non_blocking=True)
            n_acc_out_h.copy_(self.out.n_accepted, non_blocking=True)
            alpha_out_h.copy_(self.out.alpha, non_blocking=True)
        self.stream.synchronize()
