"""Seeded random shapes: every schedule bit for bit, and the oracle (GPU).

Each case draws B, G, V, the dtype, the layout, ragged draft lengths and
per-request temperatures (some exactly 0, which take the greedy steps) from a
fixed seed, runs the sampling call under the automatic policy (the resident
or the streaming cluster path, as the shape allows), on the streaming path
and on the persistent grid, requires identical outputs, and compares them
with the float64 oracle."""
import os
import random

import numpy as np
import pytest
import torch

import oracle
from parity import compare_greedy, compare_sample, PROB_RTOL
from speculative_decoding_verification_62_gb300 import binding
from speculative_decoding_verification_62_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
NTHREADS = os.cpu_count() or 1
VOCABS = [1, 7, 33, 4097, 8193, 20001, 32000, 50000]


def draw_case(i):
    r = random.Random(6200 + i)
    B = r.choice([1, 2, 3, 5, 8, 11, 15, 16, 24, 40])
    G = r.randint(0, 7)
    V = r.choice(VOCABS)
    dt = r.choice(["bf16", "f32"])
    packed = r.random() < 0.4
    temps = [0.0 if r.random() < 0.15 else round(r.uniform(0.3, 1.6), 3) for _ in range(B)]
    return B, G, V, dt, packed, temps


def run(w, packed, schedule):
    prev = binding.spec_verify_set_schedule(schedule)
    try:
        v = binding.Verifier(w.B, w.G, w.V, DEV)
        if packed:
            pk = W.pack(w)
            p = torch.full((pk.total,), float("nan"), dtype=torch.float64, device=DEV)
            q = torch.full_like(p, float("nan"))
            v.sample_packed(pk.target, pk.draft, pk.cu_draft, pk.draft_tokens, pk.uniforms,
                            pk.temperature, p, q)
            p, q = (W.unpack_per_draft(x, pk.cu_draft, w.G) for x in (p, q))
        else:
            p = torch.full((w.B, w.G), float("nan"), dtype=torch.float64, device=DEV)
            q = torch.full_like(p, float("nan"))
            v.sample(w.target, w.draft, w.draft_tokens, w.gamma, w.uniforms, w.temperature, p, q)
        torch.cuda.synchronize()
        st = binding.spec_verify_status(v.workspace)
        assert st == 0, binding.status_names(st)
        return (v.out_tokens.cpu().numpy(), v.num_accepted.cpu().numpy(), p.cpu(), q.cpu())
    finally:
        binding.spec_verify_set_schedule(prev)


@pytest.mark.parametrize("i", range(24))
def test_fuzz_sampling(i):
    B, G, V, dt, packed, temps = draw_case(i)
    w = W.make_random(B, G, V, dt, seed=100 + i, gamma="ragged", temperature=temps).to(DEV)
    a = run(w, packed, binding.SCHEDULE_AUTO)
    for sched in (binding.SCHEDULE_STREAM, binding.SCHEDULE_PERSISTENT):
        b = run(w, packed, sched)
        assert (a[0] == b[0]).all() and (a[1] == b[1]).all()
        for x, y in ((a[2], b[2]), (a[3], b[3])):
            nan = torch.isnan(y)
            assert torch.equal(torch.isnan(x), nan) and torch.equal(x[~nan], y[~nan])
    ref = oracle.sample(**W.oracle_inputs(w), nthreads=NTHREADS)
    rep = compare_sample(ref, a[0], a[1], w.gamma.cpu().numpy(), a[2].numpy(), a[3].numpy())
    assert not rep.mismatches, (draw_case(i), rep.mismatches[:3])
    assert rep.max_prob_rel_err < PROB_RTOL


@pytest.mark.parametrize("i", range(12))
def test_fuzz_greedy(i):
    B, G, V, dt, packed, _ = draw_case(100 + i)
    w = W.make_random(B, G, V, dt, seed=300 + i, gamma="ragged").to(DEV)
    if G:
        am = w.target[:, :G].float().argmax(dim=2).to(torch.int32)
        keep = torch.rand(w.draft_tokens.shape, device=DEV,
                          generator=torch.Generator(DEV).manual_seed(i)) < 0.7
        w.draft_tokens = torch.where(keep, am, w.draft_tokens).contiguous()
        for b in range(B):
            w.draft_tokens[b, int(w.gamma[b]):] = 0
    outs = []
    for sched in (binding.SCHEDULE_AUTO, binding.SCHEDULE_STREAM, binding.SCHEDULE_PERSISTENT):
        prev = binding.spec_verify_set_schedule(sched)
        try:
            v = binding.Verifier(B, G, V, DEV)
            if packed:
                pk = W.pack(w)
                v.greedy_packed(pk.target, pk.cu_draft, pk.draft_tokens)
            else:
                v.greedy(w.target, w.draft_tokens, w.gamma)
            torch.cuda.synchronize()
            assert binding.spec_verify_status(v.workspace) == 0
            outs.append((v.out_tokens.cpu().numpy(), v.num_accepted.cpu().numpy()))
        finally:
            binding.spec_verify_set_schedule(prev)
    for o in outs[1:]:
        assert (outs[0][0] == o[0]).all() and (outs[0][1] == o[1]).all()
    ref = oracle.greedy(W.logits_numpy(w.target), w.draft_tokens.cpu().numpy(), w.gamma.cpu().numpy())
    bad = compare_greedy(ref, outs[0][0], outs[0][1])
    assert not bad, bad[:3]


def test_fuzz_covers_both_cluster_paths():
    """Under the automatic policy the drawn shapes include batches on the
    resident and on the streaming cluster path (the persistent grid runs every
    case by force)."""
    routes = set()
    for i in range(24):
        B, G, V, dt, _, _ = draw_case(i)
        tdt = torch.bfloat16 if dt == "bf16" else torch.float32
        routes.add(binding.spec_verify_route(tdt, B, G, V)[0])
    assert routes == {binding.ROUTE_CLUSTER, binding.ROUTE_STREAM}


def draw_large_case(i):
    r = random.Random(9100 + i)
    B = r.choice([160, 257, 400, 640])
    G = r.randint(0, 7)
    V = r.choice([33, 4097, 8193, 20001])
    dt = r.choice(["bf16", "f32"])
    packed = r.random() < 0.4
    temps = [0.0 if r.random() < 0.1 else round(r.uniform(0.3, 1.6), 3) for _ in range(B)]
    return B, G, V, dt, packed, temps


@pytest.mark.parametrize("i", range(6))
def test_fuzz_claims_sampling(i):
    """Batches beyond one wave: request claims (longest first, ragged lengths)
    against the persistent grid and the oracle."""
    B, G, V, dt, packed, temps = draw_large_case(i)
    w = W.make_random(B, G, V, dt, seed=500 + i, gamma="ragged", temperature=temps).to(DEV)
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    assert binding.spec_verify_route(tdt, B, G, V)[0] in (binding.ROUTE_CLAIMS, binding.ROUTE_PIPELINE)
    a = run(w, packed, binding.SCHEDULE_AUTO)
    b = run(w, packed, binding.SCHEDULE_PERSISTENT)
    assert (a[0] == b[0]).all() and (a[1] == b[1]).all()
    for x, y in ((a[2], b[2]), (a[3], b[3])):
        nan = torch.isnan(y)
        assert torch.equal(torch.isnan(x), nan) and torch.equal(x[~nan], y[~nan])
    ref = oracle.sample(**W.oracle_inputs(w), nthreads=NTHREADS)
    rep = compare_sample(ref, a[0], a[1], w.gamma.cpu().numpy(), a[2].numpy(), a[3].numpy())
    assert not rep.mismatches, (draw_large_case(i)[:5], rep.mismatches[:3])
    assert rep.max_prob_rel_err < PROB_RTOL


@pytest.mark.parametrize("i", range(4))
def test_fuzz_claims_greedy(i):
    """Greedy batches beyond one wave of two CTAs per SM: request claims read
    target rows one at a time up to the first mismatch (lazily), against the
    persistent grid (every row) and the oracle.  Drafts are planted as the
    argmax with probability 0.7, so mismatches come at every position."""
    r = random.Random(9300 + i)
    B = r.choice([320, 400, 640, 1000])
    G = r.randint(0, 7)
    V = r.choice([33, 4097, 20001])
    dt = r.choice(["bf16", "f32"])
    packed = r.random() < 0.4
    w = W.make_random(B, G, V, dt, seed=700 + i, gamma="ragged").to(DEV)
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    assert binding.spec_verify_route(tdt, B, G, V, True)[0] == binding.ROUTE_CLAIMS
    if G:
        am = w.target[:, :G].float().argmax(dim=2).to(torch.int32)
        keep = torch.rand(w.draft_tokens.shape, device=DEV,
                          generator=torch.Generator(DEV).manual_seed(50 + i)) < 0.7
        w.draft_tokens = torch.where(keep, am, w.draft_tokens).contiguous()
    outs = []
    for sched in (binding.SCHEDULE_AUTO, binding.SCHEDULE_PERSISTENT):
        prev = binding.spec_verify_set_schedule(sched)
        try:
            v = binding.Verifier(B, G, V, DEV)
            if packed:
                pk = W.pack(w)
                v.greedy_packed(pk.target, pk.cu_draft, pk.draft_tokens)
            else:
                v.greedy(w.target, w.draft_tokens, w.gamma)
            torch.cuda.synchronize()
            assert binding.spec_verify_status(v.workspace) == 0
            outs.append((v.out_tokens.cpu().numpy(), v.num_accepted.cpu().numpy()))
        finally:
            binding.spec_verify_set_schedule(prev)
    assert (outs[0][0] == outs[1][0]).all() and (outs[0][1] == outs[1][1]).all()
    ref = oracle.greedy(W.logits_numpy(w.target), w.draft_tokens.cpu().numpy(),
                        w.gamma.cpu().numpy(), nthreads=NTHREADS)
    bad = compare_greedy(ref, outs[0][0], outs[0][1])
    assert not bad, bad[:3]
