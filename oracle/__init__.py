"""Float64 CPU oracle of the speculative-sampling verify step (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg are the only callers.  The CUDA product path never
imports this package, and this package imports nothing from it.

The arithmetic lives in ``spec_verify_ref.c`` (plain C, float64); this module
compiles it with gcc on first use and marshals numpy arrays.  See the C file's
header for the passages each step follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_verify_ref.c")
_LIB = os.path.join(_HERE, "libspec_verify_ref.so")
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile an oracle source file into a shared library (gcc, float64, OpenMP)."""
    stale = not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src)
    if force or stale:
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", "-Wall",
               "-Wextra", "-o", tmp, src, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _logits(a, name):
    """Accept float32 arrays, or bf16 given as uint16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.uint16:
        return a, BF16
    raise TypeError(f"{name}: expected float32 or uint16 (bf16 bits), got {a.dtype}")


class Oracle:
    """One loaded copy of the oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        vp, c_int = ctypes.c_void_p, ctypes.c_int
        lib.sv_ref_sample.restype = c_int
        lib.sv_ref_sample.argtypes = [vp, vp, c_int, c_int, c_int, c_int, vp, vp, vp, vp,
                                      vp, vp, vp, vp, vp, vp, vp, c_int, c_int]
        lib.sv_ref_greedy.restype = c_int
        lib.sv_ref_greedy.argtypes = [vp, c_int, c_int, c_int, c_int, vp, vp, vp, vp, vp,
                                      c_int]
        lib.sv_ref_softmax_row.restype = c_int
        lib.sv_ref_softmax_row.argtypes = [vp, c_int, c_int, ctypes.c_double, vp]
        self.lib = lib
        self.path = path

    def sample(self, target, draft, draft_tokens, gamma, uniforms, temperature, nthreads=0,
               rows_first=False):
        """Sampling verify step.

        target [B][G+1][V], draft [B][G][V] (float32, or uint16 bf16 bits);
        draft_tokens int32 [B][G]; gamma int32 [B]; uniforms [B][G+1] (float32 or
        float64; widened exactly); temperature float32 [B].  rows_first spreads
        the row statistics over threads before the requests (same results).

        Returns a dict with out_tokens [B][G+1], num_accepted [B], p_tok/q_tok
        [B][G], margin_accept [B][G] (NaN where not evaluated), margin_cdf [B]
        and resid_mass [B] (the float64 residual mass after a rejection, NaN
        when every draft was accepted or the request is greedy).
        """
        target, dt = _logits(target, "target")
        B, G1, V = target.shape
        G = G1 - 1
        if G > 0:
            draft, dd = _logits(draft, "draft")
            if dd != dt or draft.shape != (B, G, V):
                raise ValueError("draft must match target's dtype and have shape [B][G][V]")
        else:
            draft = np.zeros((B, 0, V), dtype=target.dtype)
        tokens = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, G)
        gamma = np.ascontiguousarray(gamma, dtype=np.int32).reshape(B)
        u = np.ascontiguousarray(uniforms, dtype=np.float64).reshape(B, G + 1)
        temp = np.ascontiguousarray(temperature, dtype=np.float32).reshape(B)
        out = np.empty((B, G + 1), dtype=np.int32)
        nacc = np.empty(B, dtype=np.int32)
        p_tok = np.empty((B, G))
        q_tok = np.empty((B, G))
        m_acc = np.empty((B, G))
        m_cdf = np.empty(B)
        mass = np.empty(B)
        rc = self.lib.sv_ref_sample(_ptr(target), _ptr(draft), dt, B, G, V, _ptr(tokens),
                                    _ptr(gamma), _ptr(u), _ptr(temp), _ptr(out), _ptr(nacc),
                                    _ptr(p_tok), _ptr(q_tok), _ptr(m_acc), _ptr(m_cdf),
                                    _ptr(mass), 1 if rows_first else 0, int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle rejected the input (code {rc})")
        return dict(out_tokens=out, num_accepted=nacc, p_tok=p_tok, q_tok=q_tok,
                    margin_accept=m_acc, margin_cdf=m_cdf, resid_mass=mass)

    def greedy(self, target, draft_tokens, gamma, nthreads=0):
        """Greedy (argmax-match) verify step: out_tokens, num_accepted, exact_tie."""
        target, dt = _logits(target, "target")
        B, G1, V = target.shape
        G = G1 - 1
        tokens = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, G)
        gamma = np.ascontiguousarray(gamma, dtype=np.int32).reshape(B)
        out = np.empty((B, G + 1), dtype=np.int32)
        nacc = np.empty(B, dtype=np.int32)
        tie = np.empty((B, G + 1), dtype=np.int32)
        rc = self.lib.sv_ref_greedy(_ptr(target), dt, B, G, V, _ptr(tokens), _ptr(gamma),
                                    _ptr(out), _ptr(nacc), _ptr(tie), int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle rejected the input (code {rc})")
        return dict(out_tokens=out, num_accepted=nacc, exact_tie=tie)

    def softmax_row(self, row, temperature):
        """Temperature softmax of one row of logits, float64."""
        row, dt = _logits(row, "row")
        V = row.shape[-1]
        p = np.empty(V)
        rc = self.lib.sv_ref_softmax_row(_ptr(row), dt, V, float(temperature), _ptr(p))
        if rc != 0:
            raise ValueError("invalid softmax input")
        return p


def default() -> Oracle:
    """The oracle built from this directory's source (compiled on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(build())
    return _lib


def sample(*args, **kwargs):
    return default().sample(*args, **kwargs)


def greedy(*args, **kwargs):
    return default().greedy(*args, **kwargs)


def softmax_row(*args, **kwargs):
    return default().softmax_row(*args, **kwargs)
