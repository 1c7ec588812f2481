"""spec_verify_sample_noalloc (built-in scratch array, no workspace) against
spec_verify_sample on the same inputs, two calls in a row.  Both entry points
run the same kernel, so tokens and accepted counts must agree exactly and the
probabilities within the parity tolerance; the file is collected last so that
it also runs after every other GPU test in the same process."""
import pytest
import torch

from speculative_decoding_verification_62_gb300 import binding
from speculative_decoding_verification_62_gb300 import workloads as W

PROB_RTOL = 1e-5

pytestmark = pytest.mark.gpu


def _with_workspace(w):
    B, G, V = w.B, w.G, w.V
    out = torch.full((B, G + 1), -7, dtype=torch.int32, device="cuda")
    nacc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    p = torch.empty((B, G), dtype=torch.float64, device="cuda")
    q = torch.empty((B, G), dtype=torch.float64, device="cuda")
    ws = binding.make_workspace(B, G, V)
    binding.spec_verify_sample(w.target, w.draft, w.draft_tokens, w.gamma, w.uniforms,
                               w.temperature, out, nacc, ws, p, q)
    torch.cuda.synchronize()
    assert binding.spec_verify_status(ws) == 0
    return out, nacc, p, q


def _noalloc(w):
    B, G = w.B, w.G
    out = torch.full((B, G + 1), -7, dtype=torch.int32, device="cuda")
    nacc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    p = torch.empty((B, G), dtype=torch.float64, device="cuda")
    q = torch.empty((B, G), dtype=torch.float64, device="cuda")
    binding.spec_verify_sample_noalloc(w.target, w.draft, w.draft_tokens, w.gamma, w.uniforms,
                                       w.temperature, out, nacc, p, q)
    torch.cuda.synchronize()
    return out, nacc, p, q


def _same(a, b):
    out_a, nacc_a, p_a, q_a = a
    out_b, nacc_b, p_b, q_b = b
    assert torch.equal(out_a, out_b)
    assert torch.equal(nacc_a, nacc_b)
    for x, y in ((p_a, p_b), (q_a, q_b)):
        nan = torch.isnan(x)
        assert torch.equal(nan, torch.isnan(y))
        assert torch.allclose(x[~nan], y[~nan], rtol=PROB_RTOL, atol=0.0)


def _case(case):
    if case == "config2":
        return W.make("2", device="cuda")
    if case == "ragged_f32":
        return W.make_random(B=37, G=5, V=20001, dtype="f32", device="cuda", seed=4242,
                             gamma="ragged", temperature=0.9)
    # the largest shape the header names as fitting the built-in scratch:
    # more requests than resident CTAs, so the streaming schedule claims them
    return W.make_random(B=512, G=3, V=128256, dtype="bf16", device="cuda", seed=4243,
                         gamma="ragged", temperature=0.8)


@pytest.mark.parametrize("schedule", ["auto", "persistent"])
@pytest.mark.parametrize("case", ["config2", "ragged_f32", "claims_512x3x128256"])
def test_noalloc_matches_workspace_entry_point_twice(case, schedule):
    w = _case(case)
    assert binding.spec_verify_workspace_size(w.B, w.G, w.V) <= binding.SV_NOALLOC_SCRATCH_BYTES
    policy = binding.SCHEDULE_AUTO if schedule == "auto" else binding.SCHEDULE_PERSISTENT
    prev = binding.spec_verify_set_schedule(policy)
    try:
        ref = _with_workspace(w)
        first = _noalloc(w)
        second = _noalloc(w)
    finally:
        binding.spec_verify_set_schedule(prev)
    _same(ref, first)
    _same(ref, second)


def test_noalloc_rejects_oversized_problem():
    w = W.make_random(B=2, G=3, V=64, dtype="bf16", device="cuda", seed=1)
    big = (4096, 7, 128256)
    assert binding.spec_verify_workspace_size(*big) > binding.SV_NOALLOC_SCRATCH_BYTES
    lib = binding.load_library()
    rc = lib.spec_verify_sample_noalloc(w.target.data_ptr(), w.draft.data_ptr(), 1, *big,
                                        w.draft_tokens.data_ptr(), w.gamma.data_ptr(),
                                        w.uniforms.data_ptr(), w.temperature.data_ptr(),
                                        w.draft_tokens.data_ptr(), w.gamma.data_ptr(), None,
                                        None, None)
    assert rc == -6
