"""The C-ABI library builds, loads, exports every declared symbol, and rejects
bad host arguments before launching anything (CPU only: no kernel runs)."""
import ctypes
import os
import re

import pytest

from speculative_decoding_verification_62_gb300 import binding

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "spec_verify.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_verify_\w+)\s*\(", text)))


def test_exports_every_declared_symbol():
    lib = binding.load_library()
    names = declared_functions()
    assert set(names) == set(binding.EXPORTS), names
    for n in names:
        assert getattr(lib, n) is not None


def header_defines():
    """SV_* constants of the header: #define lines and enumerator values."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    d = {m.group(1): int(m.group(2), 0)
         for m in re.finditer(r"^#define\s+(SV_\w+)\s+\(?(-?(?:0x[0-9a-fA-F]+|\d+))", text, re.M)}
    d.update({m.group(1): int(m.group(2), 0)
              for m in re.finditer(r"\b(SV_\w+)\s*=\s*(-?(?:0x[0-9a-fA-F]+|\d+))u?\b", text)})
    return d


def test_binding_constants_match_the_header():
    """The binding's schedule, route, dtype and status constants are the
    header's values (the binding only marshals; it must not renumber)."""
    d = header_defines()
    assert (binding.SCHEDULE_AUTO, binding.SCHEDULE_PERSISTENT, binding.SCHEDULE_STREAM) == (
        d["SV_SCHEDULE_AUTO"], d["SV_SCHEDULE_PERSISTENT"], d["SV_SCHEDULE_STREAM"])
    assert (binding.ROUTE_PERSISTENT, binding.ROUTE_CLUSTER, binding.ROUTE_STREAM, binding.ROUTE_CLAIMS,
            binding.ROUTE_PIPELINE) == (
        d["SV_ROUTE_PERSISTENT"], d["SV_ROUTE_CLUSTER"], d["SV_ROUTE_STREAM"], d["SV_ROUTE_CLAIMS"],
        d["SV_ROUTE_PIPELINE"])
    for bit, name in binding.STATUS_BITS.items():
        assert d["SV_STATUS_" + name] == bit, name
    assert binding.SV_MAX_GAMMA == d["SV_MAX_GAMMA"]
    assert (binding.SV_F32, binding.SV_BF16) == (d["SV_F32"], d["SV_BF16"])


def test_set_schedule_rejects_unknown_policies():
    prev = binding.spec_verify_set_schedule(binding.SCHEDULE_AUTO)
    try:
        for bad in (-1, 3, 99):
            with pytest.raises(binding.SpecVerifyError):
                binding.spec_verify_set_schedule(bad)
        assert binding.spec_verify_set_schedule(binding.SCHEDULE_STREAM) == binding.SCHEDULE_AUTO
        assert binding.spec_verify_set_schedule(binding.SCHEDULE_AUTO) == binding.SCHEDULE_STREAM
    finally:
        binding.spec_verify_set_schedule(prev)


def test_workspace_size():
    s = binding.spec_verify_workspace_size(8, 3, 128256)
    assert s > 0 and s % 256 == 0
    assert binding.spec_verify_workspace_size(512, 3, 128256) > s
    assert binding.spec_verify_workspace_size(-1, 3, 10) == 0
    assert binding.spec_verify_workspace_size(1, 32, 10) == 0
    assert binding.spec_verify_workspace_size(1, 3, 0) == 0
    assert binding.spec_verify_workspace_size(1, 3, (1 << 24) + 1) == 0


def _fake(addr=0x10000):
    return ctypes.c_void_p(addr)


def _sample(**over):
    lib = binding.load_library()
    B, G, V = over.pop("B", 2), over.pop("G", 3), over.pop("V", 64)
    a = dict(target=_fake(), draft=_fake(), dtype=1, B=B, G=G, V=V, tokens=_fake(),
             gamma=_fake(), u=_fake(), T=_fake(), out=_fake(), nacc=_fake(), p=None, q=None,
             ws=_fake(0x100000), ws_bytes=binding.spec_verify_workspace_size(max(B, 0), G, V),
             stream=None)
    a.update(over)
    return lib.spec_verify_sample(a["target"], a["draft"], a["dtype"], a["B"], a["G"], a["V"],
                                  a["tokens"], a["gamma"], a["u"], a["T"], a["out"], a["nacc"],
                                  a["p"], a["q"], a["ws"], a["ws_bytes"], a["stream"])


def test_host_argument_errors_return_codes_without_launch():
    assert _sample(B=-1) == -1
    assert _sample(G=-1) == -1
    assert _sample(G=32) == -1
    assert _sample(V=0) == -1
    assert _sample(dtype=7) == -1
    assert _sample(target=None) == -2
    assert _sample(draft=None) == -2
    assert _sample(tokens=None) == -2
    assert _sample(u=None) == -2
    assert _sample(out=None) == -2
    assert _sample(ws=None) == -2
    assert _sample(ws_bytes=100) == -4
    assert _sample(target=_fake(0x10001)) == -3   # bf16 needs 2-byte alignment
    assert _sample(dtype=0, draft=_fake(0x10002)) == -3  # f32 needs 4
    assert _sample(gamma=_fake(0x10002)) == -3
    assert _sample(ws=_fake(0x100010)) == -3      # workspace needs 256
    assert _sample(p=_fake(0x10004)) == -3        # float64 outputs need 8


def test_g0_needs_no_draft_and_b0_is_a_noop():
    # B == 0 returns before any CUDA call; G == 0 accepts NULL draft pointers.
    assert _sample(B=0, G=0, draft=None, tokens=None) == 0


def test_greedy_host_errors():
    lib = binding.load_library()
    ws = binding.spec_verify_workspace_size(2, 3, 64)
    call = lambda **k: lib.spec_verify_greedy(  # noqa: E731
        k.get("t", _fake()), k.get("dt", 1), k.get("B", 2), 3, 64, k.get("tok", _fake()),
        _fake(), _fake(), _fake(), _fake(0x100000), k.get("ws", ws), None)
    assert call(dt=3) == -1
    assert call(t=None) == -2
    assert call(tok=None) == -2
    assert call(ws=0) == -4
    assert call(B=0) == 0


def test_noalloc_rejects_sizes_beyond_its_scratch_without_cuda():
    lib = binding.load_library()
    f = _fake()
    call = lambda B, G, V, **k: lib.spec_verify_sample_noalloc(  # noqa: E731
        k.get("t", f), f, 1, B, G, V, f, f, f, f, f, f, None, None, None)
    too_big = (4096, 7, 128256)
    assert binding.spec_verify_workspace_size(*too_big) > binding.SV_NOALLOC_SCRATCH_BYTES
    assert call(*too_big) == -6
    assert "4 MiB" in binding.spec_verify_strerror(-6)
    assert binding.spec_verify_workspace_size(512, 3, 128256) <= binding.SV_NOALLOC_SCRATCH_BYTES
    assert call(2, 3, 64, t=None) == -2
    assert call(2, 32, 64) == -1
    assert call(0, 3, 64) == 0  # B == 0: nothing to do, no CUDA call


def test_strerror_texts():
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert binding.spec_verify_strerror(code)
    assert "unknown" in binding.spec_verify_strerror(-99)


def test_binding_refuses_cpu_tensors():
    import torch
    t = torch.zeros((1, 2, 8), dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        binding.spec_verify_greedy(t, torch.zeros((1, 1), dtype=torch.int32),
                                   torch.ones(1, dtype=torch.int32),
                                   torch.zeros((1, 2), dtype=torch.int32),
                                   torch.zeros(1, dtype=torch.int32),
                                   torch.zeros(256, dtype=torch.uint8))


def test_wait_limit_setter_returns_previous_and_zero_restores_default():
    """The wait limit is host state for later launches (no kernel runs)."""
    prev = binding.spec_verify_set_wait_limit(5_000_000)
    try:
        assert prev == 2_000_000_000
        assert binding.spec_verify_set_wait_limit(0) == 5_000_000
        assert binding.spec_verify_set_wait_limit(0) == 2_000_000_000
    finally:
        binding.spec_verify_set_wait_limit(prev)


def test_lazy_setter_returns_previous_and_rejects_other_values():
    """Position-by-position reading is on by default; the setter is host state."""
    prev = binding.spec_verify_set_lazy(True)
    try:
        assert prev is True
        assert binding.spec_verify_set_lazy(False) is True
        assert binding.spec_verify_set_lazy(True) is False
        lib = binding.load_library()
        for bad in (-1, 2, 7):
            assert lib.spec_verify_set_lazy(bad) == -1  # SV_ERR_SCALAR
        assert binding.spec_verify_set_lazy(True) is True
    finally:
        binding.spec_verify_set_lazy(prev)
