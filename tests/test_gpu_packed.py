"""Packed (varlen) layout vs the padded layout and the float64 oracle (GPU).

Both layouts run the same kernel arithmetic, and a row's results do not depend
on its address, so their outputs must agree bit for bit; the packed results
are in turn compared with the oracle."""
import os

import pytest
import torch

import oracle
from parity import compare_greedy, compare_sample, PROB_RTOL
from speculative_decoding_verification_62_gb300 import binding
from speculative_decoding_verification_62_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
NTHREADS = os.cpu_count() or 1


def run_padded(w):
    v = binding.Verifier(w.B, w.G, w.V, DEV)
    p = torch.full((w.B, w.G), float("nan"), dtype=torch.float64, device=DEV)
    q = torch.full_like(p, float("nan"))
    v.sample(w.target, w.draft, w.draft_tokens, w.gamma, w.uniforms, w.temperature, p, q)
    torch.cuda.synchronize()
    assert binding.spec_verify_status(v.workspace) == 0
    return v.out_tokens.cpu().numpy(), v.num_accepted.cpu().numpy(), p, q


def run_packed(pk, B, G, V, probs=True):
    ws = binding.make_workspace(B, G, V)
    out = torch.full((B, G + 1), -7, dtype=torch.int32, device=DEV)
    nacc = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    p = torch.full((pk.total,), float("nan"), dtype=torch.float64, device=DEV) if probs else None
    q = torch.full_like(p, float("nan")) if probs else None
    binding.spec_verify_sample_packed(pk.target, pk.draft, pk.cu_draft, pk.draft_tokens,
                                      pk.uniforms, pk.temperature, out, nacc, ws, p, q)
    torch.cuda.synchronize()
    st = binding.spec_verify_status(ws)
    return out.cpu().numpy(), nacc.cpu().numpy(), p, q, st, ws


CASES = [(7, 4, 20001, "bf16"), (9, 3, 4097, "f32"), (12, 7, 128256, "bf16"), (5, 2, 1, "f32")]


@pytest.mark.parametrize("B,G,V,dt", CASES)
def test_packed_sample_matches_padded_and_oracle(B, G, V, dt):
    temps = [0.5 + 0.1 * i for i in range(B)]
    temps[1] = 0.0  # a greedy request inside the sampling call
    w = W.make_random(B, G, V, dt, seed=B * 31 + V, gamma="ragged", temperature=temps).to(DEV)
    w.gamma[0] = 0
    w.gamma[-1] = G
    out_p, nacc_p, pp, qp = run_padded(w)
    pk = W.pack(w)
    out, nacc, p, q, st, ws = run_packed(pk, B, G, V)
    assert st == 0, binding.status_names(st)
    assert (out == out_p).all() and (nacc == nacc_p).all()
    P = W.unpack_per_draft(p, pk.cu_draft, G)
    Q = W.unpack_per_draft(q, pk.cu_draft, G)
    for a, b in ((P, pp), (Q, qp)):
        nan = torch.isnan(b)
        assert torch.equal(torch.isnan(a), nan)
        assert torch.equal(a[~nan], b[~nan])
    ref = oracle.sample(**W.oracle_inputs(w), nthreads=NTHREADS)
    rep = compare_sample(ref, out, nacc, w.gamma.cpu().numpy(), P.cpu().numpy(), Q.cpu().numpy())
    print(rep.summary())
    assert not rep.mismatches, rep.mismatches[:5]
    assert rep.max_prob_rel_err < PROB_RTOL


@pytest.mark.parametrize("B,G,V,dt", CASES)
def test_packed_greedy_matches_oracle(B, G, V, dt):
    w = W.make_random(B, G, V, dt, seed=B * 37 + V, gamma="ragged").to(DEV)
    am = w.target[:, :G].float().argmax(dim=2).to(torch.int32)
    keep = torch.rand(w.draft_tokens.shape, device=DEV) < 0.7
    w.draft_tokens = torch.where(keep, am, w.draft_tokens).contiguous()
    for b in range(B):
        w.draft_tokens[b, int(w.gamma[b]):] = 0
    pk = W.pack(w)
    ws = binding.make_workspace(B, G, V)
    out = torch.full((B, G + 1), -7, dtype=torch.int32, device=DEV)
    nacc = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    binding.spec_verify_greedy_packed(pk.target, pk.cu_draft, pk.draft_tokens, out, nacc, ws)
    torch.cuda.synchronize()
    assert binding.spec_verify_status(ws) == 0
    ref = oracle.greedy(W.logits_numpy(w.target), w.draft_tokens.cpu().numpy(),
                        w.gamma.cpu().numpy())
    bad = compare_greedy(ref, out.cpu().numpy(), nacc.cpu().numpy())
    assert not bad, bad[:5]


@pytest.mark.parametrize("sched", [binding.SCHEDULE_PERSISTENT, binding.SCHEDULE_AUTO])
def test_packed_large_batches(sched):
    """1700 requests: on the persistent grid more than one launch takes (the
    packed offsets stay global); by default, request claims."""
    B, G, V = 1700, 3, 300
    prev = binding.spec_verify_set_schedule(sched)
    try:
        w = W.make_random(B, G, V, "bf16", seed=99, gamma="ragged").to(DEV)
        out_p, nacc_p, _, _ = run_padded(w)
        out, nacc, _, _, st, _ = run_packed(W.pack(w), B, G, V)
    finally:
        binding.spec_verify_set_schedule(prev)
    assert st == 0
    assert (out == out_p).all() and (nacc == nacc_p).all()


def test_inconsistent_prefix_is_flagged_and_contained():
    """A broken cu_draft entry flags BAD_GAMMA; the requests it touches are
    verified with no drafts inside the arrays, the others are unaffected."""
    B, G, V = 8, 3, 5000
    w = W.make_random(B, G, V, "bf16", seed=7, gamma=[3, 2, 3, 1, 0, 3, 2, 3]).to(DEV)
    out_p, nacc_p, _, _ = run_padded(w)
    pk = W.pack(w)
    pk.cu_draft[3] = pk.total + 100          # requests 2 and 3 become inconsistent
    out, nacc, _, _, st, _ = run_packed(pk, B, G, V, probs=False)
    assert "BAD_GAMMA" in binding.status_names(st)
    for b in range(B):
        if b in (2, 3):
            assert nacc[b] == 0 and out[b, 0] >= 0 and (out[b, 1:] == -1).all()
        else:
            assert (out[b] == out_p[b]).all() and nacc[b] == nacc_p[b]


def test_packed_without_drafts():
    B, G, V = 6, 2, 1000
    w = W.make_random(B, G, V, "f32", seed=3, gamma=[0] * B).to(DEV)
    out_p, nacc_p, _, _ = run_padded(w)
    pk = W.pack(w)
    out, nacc, _, _, st, _ = run_packed(pk, B, G, V, probs=False)
    assert st == 0
    assert (out == out_p).all() and (nacc == 0).all()
