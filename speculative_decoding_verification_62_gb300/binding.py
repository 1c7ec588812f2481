"""Thin ctypes binding of the C ABI in include/spec_verify.h.

Argument marshalling only: every step of the verify path runs in the CUDA
library.  Functions keep the C names.  Tensors must be CUDA, contiguous and
of the documented dtype and shape; the call is issued on the current torch
stream unless `stream` is given.  There is no CPU fallback: if the library
cannot be loaded or built, the first call raises.
"""
from __future__ import annotations

import ctypes
import threading

import torch

from . import build as _build

SV_F32, SV_BF16 = 0, 1
SV_MAX_GAMMA = 31
SV_MAX_VOCAB = 1 << 24
STATUS_BITS = {1: "BAD_GAMMA", 2: "BAD_TOKEN", 4: "BAD_UNIFORM", 8: "BAD_TEMPERATURE",
               16: "NONFINITE_ROW", 32: "INTERNAL", 64: "TIMEOUT"}
SV_NOALLOC_SCRATCH_BYTES = 4 << 20
EXPORTS = ("spec_verify_workspace_size", "spec_verify_sample", "spec_verify_greedy",
           "spec_verify_sample_packed", "spec_verify_greedy_packed", "spec_verify_draw",
           "spec_verify_sample_noalloc", "spec_verify_status", "spec_verify_strerror",
           "spec_verify_set_schedule", "spec_verify_route", "spec_verify_cluster_size",
           "spec_verify_set_wait_limit", "spec_verify_set_lazy")
SCHEDULE_AUTO, SCHEDULE_PERSISTENT, SCHEDULE_STREAM = 0, 1, 2
ROUTE_PERSISTENT, ROUTE_CLUSTER, ROUTE_STREAM, ROUTE_CLAIMS, ROUTE_PIPELINE = 0, 1, 2, 3, 4

_lock = threading.Lock()
_lib = None


class SpecVerifyError(RuntimeError):
    def __init__(self, code: int):
        super().__init__(f"{spec_verify_strerror(code)} (code {code})")
        self.code = code


def load_library():
    """Load (building first if needed) libspec_verify.so and declare signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(_build.build())
        vp, ci, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        lib.spec_verify_workspace_size.restype = sz
        lib.spec_verify_workspace_size.argtypes = [ci, ci, ci]
        lib.spec_verify_sample.restype = ci
        lib.spec_verify_sample.argtypes = [vp, vp, ci, ci, ci, ci, vp, vp, vp, vp, vp, vp, vp,
                                           vp, vp, sz, vp]
        lib.spec_verify_greedy.restype = ci
        lib.spec_verify_greedy.argtypes = [vp, ci, ci, ci, ci, vp, vp, vp, vp, vp, sz, vp]
        lib.spec_verify_sample_packed.restype = ci
        lib.spec_verify_sample_packed.argtypes = [vp, vp, ci, ci, ci, ci, vp, ci, vp, vp, vp,
                                                  vp, vp, vp, vp, vp, sz, vp]
        lib.spec_verify_greedy_packed.restype = ci
        lib.spec_verify_greedy_packed.argtypes = [vp, ci, ci, ci, ci, vp, ci, vp, vp, vp, vp,
                                                  sz, vp]
        lib.spec_verify_draw.restype = ci
        lib.spec_verify_draw.argtypes = [vp, ci, ci, ci, vp, vp, vp, vp, sz, vp]
        lib.spec_verify_sample_noalloc.restype = ci
        lib.spec_verify_sample_noalloc.argtypes = [vp, vp, ci, ci, ci, ci, vp, vp, vp, vp, vp,
                                                   vp, vp, vp, vp]
        lib.spec_verify_status.restype = ci
        lib.spec_verify_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
        lib.spec_verify_strerror.restype = ctypes.c_char_p
        lib.spec_verify_strerror.argtypes = [ci]
        lib.spec_verify_set_schedule.restype = ci
        lib.spec_verify_set_schedule.argtypes = [ci]
        lib.spec_verify_route.restype = ci
        lib.spec_verify_route.argtypes = [ci, ci, ci, ci, ci, ctypes.POINTER(ci)]
        lib.spec_verify_cluster_size.restype = ci
        lib.spec_verify_cluster_size.argtypes = [ci, ci, ci, ci, ci]
        lib.spec_verify_set_wait_limit.restype = ctypes.c_ulonglong
        lib.spec_verify_set_wait_limit.argtypes = [ctypes.c_ulonglong]
        lib.spec_verify_set_lazy.restype = ci
        lib.spec_verify_set_lazy.argtypes = [ci]
        _lib = lib
        return lib


def spec_verify_strerror(code: int) -> str:
    return load_library().spec_verify_strerror(int(code)).decode()


def spec_verify_set_schedule(schedule: int) -> int:
    """SCHEDULE_AUTO, SCHEDULE_PERSISTENT or SCHEDULE_STREAM for the calls that follow;
    returns the previous policy."""
    rc = load_library().spec_verify_set_schedule(int(schedule))
    if rc < 0:
        raise SpecVerifyError(rc)
    return rc


def spec_verify_set_lazy(on: bool) -> bool:
    """Position-by-position reading on the request-claims schedule for the calls
    that follow (the default); returns the previous setting."""
    rc = load_library().spec_verify_set_lazy(1 if on else 0)
    if rc < 0:
        raise SpecVerifyError(rc)
    return bool(rc)


def spec_verify_set_wait_limit(ns: int) -> int:
    """Limit (ns) of every bounded wait in later calls (0: the 2 s default);
    returns the previous limit."""
    return int(load_library().spec_verify_set_wait_limit(int(ns)))


def spec_verify_route(dtype: torch.dtype, B: int, G: int, V: int, greedy: bool = False):
    """(ROUTE_*, CTAs per request) of the kernel a call of this shape would use."""
    code = SV_BF16 if dtype == torch.bfloat16 else SV_F32
    C = ctypes.c_int(0)
    rc = load_library().spec_verify_route(code, int(B), int(G), int(V), int(bool(greedy)),
                                          ctypes.byref(C))
    if rc < 0:
        raise SpecVerifyError(rc)
    return rc, C.value


def spec_verify_cluster_size(dtype: torch.dtype, B: int, G: int, V: int, greedy: bool = False) -> int:
    """CTAs per request of the cluster schedule (resident, streaming; 1 for request claims)
    for this shape, 0 for the persistent grid."""
    code = SV_BF16 if dtype == torch.bfloat16 else SV_F32
    rc = load_library().spec_verify_cluster_size(code, int(B), int(G), int(V), int(bool(greedy)))
    if rc < 0:
        raise SpecVerifyError(rc)
    return rc


def spec_verify_workspace_size(B: int, G: int, V: int) -> int:
    return int(load_library().spec_verify_workspace_size(int(B), int(G), int(V)))


def make_workspace(B: int, G: int, V: int, device="cuda") -> torch.Tensor:
    """Zero-filled device workspace (256-byte aligned by the caching allocator)."""
    n = spec_verify_workspace_size(B, G, V)
    if n == 0:
        raise ValueError(f"invalid sizes B={B} G={G} V={V}")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SV_BF16
    if t.dtype == torch.float32:
        return SV_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _dev(t, name, dtype=None, shape=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return ctypes.c_void_p(t.data_ptr()) if t.numel() else ctypes.c_void_p(0)


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def spec_verify_sample(target_logits, draft_logits, draft_tokens, gamma, uniforms, temperature,
                       out_tokens, num_accepted, workspace, p_tok=None, q_tok=None,
                       stream=None) -> None:
    """Sampling verify step; see include/spec_verify.h for the contract."""
    B, G1, V = target_logits.shape
    G = G1 - 1
    code = _dtype_code(target_logits)
    args = (
        _dev(target_logits, "target_logits"),
        _dev(draft_logits, "draft_logits", target_logits.dtype, (B, G, V)),
        code, B, G, V,
        _dev(draft_tokens, "draft_tokens", torch.int32, (B, G)),
        _dev(gamma, "gamma", torch.int32, (B,)),
        _dev(uniforms, "uniforms", torch.float32, (B, G + 1)),
        _dev(temperature, "temperature", torch.float32, (B,)),
        _dev(out_tokens, "out_tokens", torch.int32, (B, G + 1)),
        _dev(num_accepted, "num_accepted", torch.int32, (B,)),
        _dev(p_tok, "p_tok", torch.float64, (B, G)),
        _dev(q_tok, "q_tok", torch.float64, (B, G)),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    rc = load_library().spec_verify_sample(*args)
    if rc != 0:
        raise SpecVerifyError(rc)


def spec_verify_sample_packed(target_logits, draft_logits, cu_draft, draft_tokens, uniforms,
                              temperature, out_tokens, num_accepted, workspace, p_tok=None,
                              q_tok=None, stream=None) -> None:
    """Sampling verify step on the packed layout; see include/spec_verify.h."""
    B = cu_draft.numel() - 1
    total = draft_tokens.numel()
    V = target_logits.shape[1]
    G = out_tokens.shape[1] - 1
    if target_logits.shape[0] != total + B:
        raise ValueError("target_logits must have total_drafts + B rows")
    code = _dtype_code(target_logits)
    args = (
        _dev(target_logits, "target_logits"),
        _dev(draft_logits, "draft_logits", target_logits.dtype, (total, V)),
        code, B, G, V,
        _dev(cu_draft, "cu_draft", torch.int32, (B + 1,)), total,
        _dev(draft_tokens, "draft_tokens", torch.int32, (total,)),
        _dev(uniforms, "uniforms", torch.float32, (total + B,)),
        _dev(temperature, "temperature", torch.float32, (B,)),
        _dev(out_tokens, "out_tokens", torch.int32, (B, G + 1)),
        _dev(num_accepted, "num_accepted", torch.int32, (B,)),
        _dev(p_tok, "p_tok", torch.float64, (total,)),
        _dev(q_tok, "q_tok", torch.float64, (total,)),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    rc = load_library().spec_verify_sample_packed(*args)
    if rc != 0:
        raise SpecVerifyError(rc)


def spec_verify_greedy_packed(target_logits, cu_draft, draft_tokens, out_tokens, num_accepted,
                              workspace, stream=None) -> None:
    """Greedy verify step on the packed layout; see include/spec_verify.h."""
    B = cu_draft.numel() - 1
    total = draft_tokens.numel()
    V = target_logits.shape[1]
    G = out_tokens.shape[1] - 1
    if target_logits.shape[0] != total + B:
        raise ValueError("target_logits must have total_drafts + B rows")
    args = (
        _dev(target_logits, "target_logits"), _dtype_code(target_logits), B, G, V,
        _dev(cu_draft, "cu_draft", torch.int32, (B + 1,)), total,
        _dev(draft_tokens, "draft_tokens", torch.int32, (total,)),
        _dev(out_tokens, "out_tokens", torch.int32, (B, G + 1)),
        _dev(num_accepted, "num_accepted", torch.int32, (B,)),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    rc = load_library().spec_verify_greedy_packed(*args)
    if rc != 0:
        raise SpecVerifyError(rc)


def spec_verify_draw(logits, uniforms, temperature, tokens, workspace, stream=None) -> None:
    """One token per row from softmax(logits / T) by inverse CDF (argmax at T = 0)."""
    B, V = logits.shape
    args = (
        _dev(logits, "logits"), _dtype_code(logits), B, V,
        _dev(uniforms, "uniforms", torch.float32, (B,)),
        _dev(temperature, "temperature", torch.float32, (B,)),
        _dev(tokens, "tokens", torch.int32, (B,)),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    rc = load_library().spec_verify_draw(*args)
    if rc != 0:
        raise SpecVerifyError(rc)


def spec_verify_sample_noalloc(target_logits, draft_logits, draft_tokens, gamma, uniforms,
                               temperature, out_tokens, num_accepted, p_tok=None, q_tok=None,
                               stream=None) -> None:
    """Sampling verify step on the library's built-in scratch array (no workspace)."""
    B, G1, V = target_logits.shape
    G = G1 - 1
    code = _dtype_code(target_logits)
    args = (
        _dev(target_logits, "target_logits"),
        _dev(draft_logits, "draft_logits", target_logits.dtype, (B, G, V)),
        code, B, G, V,
        _dev(draft_tokens, "draft_tokens", torch.int32, (B, G)),
        _dev(gamma, "gamma", torch.int32, (B,)),
        _dev(uniforms, "uniforms", torch.float32, (B, G + 1)),
        _dev(temperature, "temperature", torch.float32, (B,)),
        _dev(out_tokens, "out_tokens", torch.int32, (B, G + 1)),
        _dev(num_accepted, "num_accepted", torch.int32, (B,)),
        _dev(p_tok, "p_tok", torch.float64, (B, G)),
        _dev(q_tok, "q_tok", torch.float64, (B, G)),
        _stream(stream))
    rc = load_library().spec_verify_sample_noalloc(*args)
    if rc != 0:
        raise SpecVerifyError(rc)


def spec_verify_greedy(target_logits, draft_tokens, gamma, out_tokens, num_accepted, workspace,
                       stream=None) -> None:
    """Greedy (argmax-match) verify step; see include/spec_verify.h."""
    B, G1, V = target_logits.shape
    G = G1 - 1
    args = (
        _dev(target_logits, "target_logits"), _dtype_code(target_logits), B, G, V,
        _dev(draft_tokens, "draft_tokens", torch.int32, (B, G)),
        _dev(gamma, "gamma", torch.int32, (B,)),
        _dev(out_tokens, "out_tokens", torch.int32, (B, G + 1)),
        _dev(num_accepted, "num_accepted", torch.int32, (B,)),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    rc = load_library().spec_verify_greedy(*args)
    if rc != 0:
        raise SpecVerifyError(rc)


def spec_verify_status(workspace, stream=None) -> int:
    """Read and clear the workspace status word (synchronises the stream)."""
    out = ctypes.c_uint32(0)
    rc = load_library().spec_verify_status(_dev(workspace, "workspace", torch.uint8),
                                           _stream(stream), ctypes.byref(out))
    if rc != 0:
        raise SpecVerifyError(rc)
    return int(out.value)


def status_names(bits: int) -> list[str]:
    return [n for b, n in STATUS_BITS.items() if bits & b]


class Verifier:
    """Owns output buffers and a workspace for one (B, G, V) shape on one device."""

    def __init__(self, B: int, G: int, V: int, device="cuda"):
        self.B, self.G, self.V = B, G, V
        self.workspace = make_workspace(B, G, V, device)
        self.out_tokens = torch.empty((B, G + 1), dtype=torch.int32, device=device)
        self.num_accepted = torch.empty((B,), dtype=torch.int32, device=device)

    def sample(self, target, draft, draft_tokens, gamma, uniforms, temperature, p_tok=None,
               q_tok=None, stream=None):
        spec_verify_sample(target, draft, draft_tokens, gamma, uniforms, temperature,
                           self.out_tokens, self.num_accepted, self.workspace, p_tok, q_tok,
                           stream)
        return self.out_tokens, self.num_accepted

    def greedy(self, target, draft_tokens, gamma, stream=None):
        spec_verify_greedy(target, draft_tokens, gamma, self.out_tokens, self.num_accepted,
                           self.workspace, stream)
        return self.out_tokens, self.num_accepted

    def sample_packed(self, target, draft, cu_draft, draft_tokens, uniforms, temperature,
                      p_tok=None, q_tok=None, stream=None):
        spec_verify_sample_packed(target, draft, cu_draft, draft_tokens, uniforms, temperature,
                                  self.out_tokens, self.num_accepted, self.workspace, p_tok,
                                  q_tok, stream)
        return self.out_tokens, self.num_accepted

    def greedy_packed(self, target, cu_draft, draft_tokens, stream=None):
        spec_verify_greedy_packed(target, cu_draft, draft_tokens, self.out_tokens,
                                  self.num_accepted, self.workspace, stream)
        return self.out_tokens, self.num_accepted
