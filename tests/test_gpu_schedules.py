"""The three schedules against each other and the oracle (GPU).

The resident cluster path (small batches), the streaming cluster path
(batches of up to one cluster per SM) and the persistent grid compute every
value with the same arithmetic, so their outputs must agree bit for bit; the
results are also compared with the float64 oracle."""
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
SCHEDULES = (binding.SCHEDULE_AUTO, binding.SCHEDULE_STREAM, binding.SCHEDULE_PERSISTENT)


def sample_all(w, probs=True, packed=False):
    """[auto, stream, persistent] results, each (out, nacc, p, q)."""
    res = []
    for sched in SCHEDULES:
        prev = binding.spec_verify_set_schedule(sched)
        try:
            v = binding.Verifier(w.B, w.G, w.V, DEV)
            if packed:
                pk = W.pack(w)
                p = torch.full((pk.total,), float("nan"), dtype=torch.float64, device=DEV) if probs else None
                q = torch.full_like(p, float("nan")) if probs else None
                v.sample_packed(pk.target, pk.draft, pk.cu_draft, pk.draft_tokens, pk.uniforms,
                                pk.temperature, p, q)
                if probs:
                    p, q = (W.unpack_per_draft(x, pk.cu_draft, w.G) for x in (p, q))
            else:
                p = torch.full((w.B, w.G), float("nan"), dtype=torch.float64, device=DEV) if probs else None
                q = torch.full_like(p, float("nan")) if probs else None
                v.sample(w.target, w.draft, w.draft_tokens, w.gamma, w.uniforms, w.temperature, p, q)
            torch.cuda.synchronize()
            st = binding.spec_verify_status(v.workspace)
            assert st == 0, binding.status_names(st)
            res.append((v.out_tokens.cpu().numpy(), v.num_accepted.cpu().numpy(),
                        None if p is None else p.cpu(), None if q is None else q.cpu()))
        finally:
            binding.spec_verify_set_schedule(prev)
    return res


def route(dt, B, G, V, greedy=False, sched=binding.SCHEDULE_AUTO):
    prev = binding.spec_verify_set_schedule(sched)
    try:
        return binding.spec_verify_route(dt, B, G, V, greedy)
    finally:
        binding.spec_verify_set_schedule(prev)


def same(a, b):
    (oa, na, pa, qa), (ob, nb, pb, qb) = a, b
    assert (oa == ob).all() and (na == nb).all()
    for x, y in ((pa, pb), (qa, qb)):
        if x is None:
            continue
        nan = torch.isnan(y)
        assert torch.equal(torch.isnan(x), nan)
        assert torch.equal(x[~nan], y[~nan])


def all_same(res):
    for r in res[1:]:
        same(res[0], r)


def against_oracle(w, res):
    out, nacc, p, q = res
    ref = oracle.sample(**W.oracle_inputs(w), nthreads=NTHREADS)
    rep = compare_sample(ref, out, nacc, w.gamma.cpu().numpy(),
                         None if p is None else p.numpy(), None if q is None else q.numpy())
    print(w.name, rep.summary())
    assert not rep.mismatches, rep.mismatches[:5]
    assert rep.max_prob_rel_err < PROB_RTOL


def test_routes():
    """Resident clusters while a request's units fit one cluster's warps and the
    batch one wave; streaming clusters up to one cluster per SM; the
    persistent grid beyond."""
    bf, f32 = torch.bfloat16, torch.float32
    R, S, P = binding.ROUTE_CLUSTER, binding.ROUTE_STREAM, binding.ROUTE_PERSISTENT
    Q, L = binding.ROUTE_CLAIMS, binding.ROUTE_PIPELINE
    for dt in (bf, f32):
        assert route(dt, 1, 4, 32000)[0] == R
        assert route(dt, 8, 3, 32000)[0] == R
        assert route(dt, 512, 3, 128256) == (L, 1)  # sampled, two requests or more per SM
        assert route(dt, 200, 3, 128256) == (Q, 1)
        # a claim order too large for shared memory: the persistent grid
        assert route(dt, 100000, 3, 32000) == (P, 0)
    assert route(bf, 8, 3, 128256)[0] == R
    assert route(bf, 8, 3, 128256, greedy=True)[0] == R
    # too many units per request for one resident cluster: streaming
    kind, C = route(f32, 2, 3, 128256)
    assert kind == S and C >= 8
    assert route(bf, 2, 31, 128256)[0] == S
    kind, C = route(bf, 64, 5, 152064)
    assert kind == S and C >= 2
    # the policies
    assert route(bf, 8, 3, 128256, sched=binding.SCHEDULE_STREAM)[0] == S
    assert route(bf, 8, 3, 128256, sched=binding.SCHEDULE_PERSISTENT) == (P, 0)
    # beyond one cluster per SM: claims in both modes (sampled: the pipeline
    # when positions are read lazily)
    assert route(bf, 512, 3, 128256, greedy=True) == (Q, 1)
    assert route(bf, 512, 3, 128256, sched=binding.SCHEDULE_STREAM) == (Q, 1)
    prev = binding.spec_verify_set_lazy(False)
    try:
        assert route(bf, 512, 3, 128256) == (Q, 1)
    finally:
        binding.spec_verify_set_lazy(prev)
    assert route(bf, 512, 3, 128256, sched=binding.SCHEDULE_PERSISTENT) == (P, 0)
    assert binding.spec_verify_cluster_size(bf, 512, 3, 128256) == 1
    assert binding.spec_verify_cluster_size(bf, 8, 3, 128256) == route(bf, 8, 3, 128256)[1]


CASES = [(8, 3, 128256, "bf16"), (5, 4, 20001, "bf16"), (3, 2, 4097, "f32"), (1, 4, 32000, "f32"),
         (6, 7, 8193, "bf16"), (4, 3, 1, "bf16"), (7, 4, 152064, "bf16"), (2, 3, 32000, "f32")]


@pytest.mark.parametrize("B,G,V,dt", CASES)
def test_schedules_sample_match_each_other_and_oracle(B, G, V, dt):
    temps = [0.6 + 0.15 * i for i in range(B)]
    w = W.make_random(B, G, V, dt, seed=B * 101 + V, gamma="ragged", temperature=temps).to(DEV)
    assert binding.spec_verify_cluster_size(w.target.dtype, B, G, V) > 0
    res = sample_all(w)
    all_same(res)
    against_oracle(w, res[0])


@pytest.mark.parametrize("name", ["2", "3"])
def test_schedules_full_size(name):
    """Config 2 (B=8) on the resident path, config 3 (B=64, gamma=5,
    V=152064) on the streaming path, each against the other schedules."""
    w = W.make(name, device=DEV)
    kind = binding.spec_verify_route(w.target.dtype, w.B, w.G, w.V)[0]
    assert kind == (binding.ROUTE_CLUSTER if name == "2" else binding.ROUTE_STREAM)
    res = sample_all(w)
    all_same(res)
    against_oracle(w, res[0])


def test_cluster_zero_temperature_and_packed():
    B, G, V = 6, 4, 30001
    temps = [0.0, 0.8, 1.3, 0.0, 0.5, 1.0]
    w = W.make_random(B, G, V, "bf16", seed=5, gamma=[4, 0, 2, 3, 4, 1], temperature=temps).to(DEV)
    res = sample_all(w)
    all_same(res)
    against_oracle(w, res[0])
    resp = sample_all(w, packed=True)
    all_same(resp)
    same(res[0], resp[0])


def test_cluster_rejections_and_bonus_both_occur():
    """Sharp rows with far-off drafts reject; identical rows accept (bonus)."""
    B, G, V = 8, 3, 50000
    w = W.make_random(B, G, V, "bf16", seed=9, sigma_t=4.0, sigma_d=3.0).to(DEV)
    w.draft[::2] = w.target[::2, :G]  # even requests: q == p, every draft accepted
    res = sample_all(w)
    all_same(res)
    nacc = res[0][1]
    assert (nacc[::2] == G).all() and (nacc[1::2] < G).any()
    against_oracle(w, res[0])


@pytest.mark.parametrize("B,G,V,dt", [(8, 3, 128256, "bf16"), (5, 6, 20001, "f32"), (2, 0, 7, "bf16"),
                                      (300, 3, 20001, "bf16"), (900, 2, 4097, "f32")])
def test_schedules_greedy_match_each_other_and_oracle(B, G, V, dt):
    w = W.make_random(B, G, V, dt, seed=B + V, gamma="ragged").to(DEV)
    if G:
        am = w.target[:, :G].float().argmax(dim=2).to(torch.int32)
        keep = torch.rand(w.draft_tokens.shape, device=DEV) < 0.7
        w.draft_tokens = torch.where(keep, am, w.draft_tokens).contiguous()
        for b in range(B):
            w.draft_tokens[b, int(w.gamma[b]):] = 0
    outs = []
    for sched in SCHEDULES:
        prev = binding.spec_verify_set_schedule(sched)
        try:
            v = binding.Verifier(B, G, V, DEV)
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
    assert not bad, bad[:5]


def test_cluster_draft_sampler_matches_persistent():
    B, V = 12, 128256
    w = W.make_random(B, 0, V, "bf16", seed=17, temperature=[0.7 + 0.05 * i for i in range(B)])
    w.temperature[::5] = 0.0
    w = w.to(DEV)
    logits, u = w.target[:, 0].contiguous(), w.uniforms[:, 0].contiguous()
    toks = []
    for sched in SCHEDULES:
        prev = binding.spec_verify_set_schedule(sched)
        try:
            t = torch.full((B,), -5, dtype=torch.int32, device=DEV)
            ws = binding.make_workspace(B, 0, V)
            binding.spec_verify_draw(logits, u, w.temperature, t, ws)
            torch.cuda.synchronize()
            assert binding.spec_verify_status(ws) == 0
            toks.append(t.cpu())
        finally:
            binding.spec_verify_set_schedule(prev)
    assert torch.equal(toks[0], toks[1]) and torch.equal(toks[0], toks[2])


@pytest.mark.parametrize("sched", [binding.SCHEDULE_AUTO, binding.SCHEDULE_STREAM])
def test_cluster_status_flags_and_reuse(sched):
    """Invalid device values are flagged on the cluster paths too; repeated
    calls on one workspace keep it usable."""
    B, G, V = 4, 3, 5000
    prev = binding.spec_verify_set_schedule(sched)
    try:
        w = W.make_random(B, G, V, "bf16", seed=23).to(DEV)
        w.gamma[1] = G + 5
        w.draft_tokens[2, 0] = V + 3
        v = binding.Verifier(B, G, V, DEV)
        v.sample(w.target, w.draft, w.draft_tokens, w.gamma, w.uniforms, w.temperature)
        torch.cuda.synchronize()
        names = binding.status_names(binding.spec_verify_status(v.workspace))
        assert "BAD_GAMMA" in names and "BAD_TOKEN" in names
        w2 = W.make_random(B, G, V, "bf16", seed=24).to(DEV)
        for _ in range(3):
            v.sample(w2.target, w2.draft, w2.draft_tokens, w2.gamma, w2.uniforms, w2.temperature)
        torch.cuda.synchronize()
        assert binding.spec_verify_status(v.workspace) == 0
    finally:
        binding.spec_verify_set_schedule(prev)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_vanished_residual_falls_back_to_p_on_every_schedule(dt):
    """A clear rejection whose residual mass is below the fixed-point
    resolution: the drafted token x has q(x) = 2 p(x) with p(x) ~ e^-40 and
    the target and draft rows agree elsewhere, so u = 0.9 rejects (ratio 1/2)
    while sum max(0, p - q) ~ p(x) rounds to 0 in units of 2^-39.  Both
    schedules then draw from p_k; their tokens must agree, and the token must
    have p > 0.  Against the oracle the acceptance decisions agree exactly
    and the draw is a residual-mass near tie (float64 mass below 1e-6: the
    residual is cancellation noise), counted by the comparison."""
    B, G, V = 3, 1, 4096
    w = W.make_random(B, G, V, dt, seed=31, sigma_t=1.0, sigma_d=0.0)
    x = 17
    w.target[:, 0, x] = -40.0
    w.draft[:, 0] = w.target[:, 0]
    w.draft[:, 0, x] = -40.0 + 0.6931471805599453
    w.draft_tokens[:, 0] = x
    w.uniforms[:, 0] = 0.9
    w.temperature[:] = 1.0
    w = w.to(DEV)
    res = sample_all(w, probs=False)
    assert binding.spec_verify_cluster_size(w.target.dtype, B, G, V) > 0
    all_same(res)
    out, nacc = res[0][0], res[0][1]
    assert (nacc == 0).all()
    p = torch.softmax(w.target[:, 0].double(), dim=1).cpu()
    for b in range(B):
        assert 0 <= out[b, 0] < V and out[b, 0] != x and p[b, out[b, 0]] > 0
        assert out[b, 1] == -1
    ref = oracle.sample(**W.oracle_inputs(w))
    rep = compare_sample(ref, out, nacc, w.gamma.cpu().numpy())
    assert not rep.mismatches, rep.mismatches
    assert rep.near_tie_resid == B and (ref["resid_mass"] < 1e-6).all(), ref["resid_mass"]


def test_batches_at_the_wave_limits():
    """The largest batch that fits one wave of resident clusters runs on the
    resident path and one more request on the streaming path; the largest
    batch of one streaming wave (one cluster per SM at least) and one more
    (claims).  Each matches the other schedules and the oracle."""
    G, V, bf = 2, 32000, torch.bfloat16
    kinds = {B: binding.spec_verify_route(bf, B, G, V)[0] for B in range(1, 161)}
    res_limit = max(B for B, k in kinds.items() if k == binding.ROUTE_CLUSTER)
    str_limit = max(B for B, k in kinds.items() if k == binding.ROUTE_STREAM)
    assert kinds[res_limit + 1] == binding.ROUTE_STREAM
    assert kinds[str_limit + 1] == binding.ROUTE_CLAIMS
    assert str_limit >= 64
    for B in (res_limit, res_limit + 1, str_limit, str_limit + 1):
        w = W.make_random(B, G, V, "bf16", seed=B, gamma="ragged",
                          temperature=[0.7 + 0.002 * i for i in range(B)]).to(DEV)
        res = sample_all(w)
        all_same(res)
        against_oracle(w, res[0])


@pytest.mark.parametrize("B,G,V,dt", [(300, 3, 20001, "bf16"), (200, 5, 4097, "f32"), (400, 1, 32000, "bf16"),
                                      (1000, 3, 4097, "f32"), (700, 0, 33, "bf16")])
def test_claimed_requests_match_other_schedules_and_oracle(B, G, V, dt):
    """More requests than SMs on the streaming path: two CTAs per SM, each
    taking requests in turn from a claim counter once the batch exceeds them
    (B = 400, 700, 1000; at 200 and 300 each CTA takes one).  Repeated calls on
    one workspace, then a persistent call on it, give the same results (the
    counter is reset)."""
    temps = [0.0 if i % 7 == 3 else 0.5 + 0.004 * i for i in range(B)]
    w = W.make_random(B, G, V, dt, seed=B + G, gamma="ragged", temperature=temps).to(DEV)
    assert route(w.target.dtype, B, G, V, sched=binding.SCHEDULE_STREAM) in \
        ((binding.ROUTE_CLAIMS, 1), (binding.ROUTE_PIPELINE, 1))
    res = sample_all(w)
    all_same(res)
    against_oracle(w, res[1])
    resp = sample_all(w, packed=True)  # the packed layout on every schedule
    all_same(resp)
    same(res[0], resp[0])
    v = binding.Verifier(B, G, V, DEV)
    outs = []
    for sched in (binding.SCHEDULE_STREAM, binding.SCHEDULE_STREAM, binding.SCHEDULE_PERSISTENT):
        prev = binding.spec_verify_set_schedule(sched)
        try:
            v.sample(w.target, w.draft, w.draft_tokens, w.gamma, w.uniforms, w.temperature)
            torch.cuda.synchronize()
            assert binding.spec_verify_status(v.workspace) == 0
            outs.append((v.out_tokens.cpu().numpy().copy(), v.num_accepted.cpu().numpy().copy()))
        finally:
            binding.spec_verify_set_schedule(prev)
    for o in outs:
        assert (o[0] == res[0][0]).all() and (o[1] == res[0][1]).all()


def _claims_call(w, lazy, sched=binding.SCHEDULE_STREAM):
    """One request-claims call with p/q, read lazily or eagerly (on the
    streaming kernel, or with the automatic schedule the pipeline kernel)."""
    prev_l = binding.spec_verify_set_lazy(lazy)
    prev_s = binding.spec_verify_set_schedule(sched)
    try:
        v = binding.Verifier(w.B, w.G, w.V, DEV)
        p = torch.full((w.B, w.G), float("nan"), dtype=torch.float64, device=DEV)
        q = torch.full_like(p, float("nan"))
        v.sample(w.target, w.draft, w.draft_tokens, w.gamma, w.uniforms, w.temperature, p, q)
        torch.cuda.synchronize()
        st = binding.spec_verify_status(v.workspace)
        assert st == 0, binding.status_names(st)
        return (v.out_tokens.cpu().numpy(), v.num_accepted.cpu().numpy(), p.cpu(), q.cpu())
    finally:
        binding.spec_verify_set_schedule(prev_s)
        binding.spec_verify_set_lazy(prev_l)


@pytest.mark.parametrize("B,G,V,dt,sigma_d", [(320, 7, 20001, "bf16", 0.3), (320, 7, 20001, "bf16", 2.0),
                                              (400, 1, 32000, "f32", 1.0), (500, 3, 4097, "bf16", 0.5),
                                              (600, 0, 33, "bf16", 1.0)])
def test_lazy_and_eager_reads_agree(B, G, V, dt, sigma_d):
    """Request claims read a sampled request position by position (lazily) by
    default: a position's rows are reduced and its draft tested before the
    next position is read (on the streaming kernel, and on the pipeline kernel
    that keeps two requests in flight per CTA).
    Reading every row first (eagerly) must give the same outputs bit for bit,
    p/q included (NaN past the first rejection on both); both against the
    oracle.  Lazy reads apply from two requests per CTA (B >= 304 on 152
    SMs), and not to a request holding 80 % of a CTA's share of the rows
    (gamma 7 here), so the batches mix both.  High and low acceptance (draft
    noise 0.3 and 2.0) exercise many and few lazy stages; temperature 0
    requests take the greedy steps."""
    temps = [0.0 if i % 11 == 5 else 0.6 + 0.003 * i for i in range(B)]
    w = W.make_random(B, G, V, dt, seed=77 * B + G, gamma="ragged", temperature=temps,
                      sigma_d=sigma_d).to(DEV)
    # the streaming kernel's claims, lazily and eagerly, and (automatic
    # schedule) the pipeline kernel
    assert route(w.target.dtype, B, G, V, sched=binding.SCHEDULE_STREAM) == (binding.ROUTE_CLAIMS, 1)
    assert route(w.target.dtype, B, G, V) == (binding.ROUTE_PIPELINE, 1)
    lazy = _claims_call(w, True)
    eager = _claims_call(w, False)
    piped = _claims_call(w, True, binding.SCHEDULE_AUTO)
    same(lazy, eager)
    same(piped, eager)
    against_oracle(w, piped)
    if G > 0:  # rejections and full acceptances both occur: both lazy exits run
        n, g = lazy[1], w.gamma.cpu().numpy()
        assert (n < g).any() and (n == g).any()


def _claims_greedy(w, tokens, lazy):
    prev_l = binding.spec_verify_set_lazy(lazy)
    prev_s = binding.spec_verify_set_schedule(binding.SCHEDULE_STREAM)
    try:
        v = binding.Verifier(w.B, w.G, w.V, DEV)
        v.greedy(w.target, tokens, w.gamma)
        torch.cuda.synchronize()
        st = binding.spec_verify_status(v.workspace)
        assert st == 0, binding.status_names(st)
        return v.out_tokens.cpu().numpy(), v.num_accepted.cpu().numpy()
    finally:
        binding.spec_verify_set_schedule(prev_s)
        binding.spec_verify_set_lazy(prev_l)


@pytest.mark.parametrize("B,G,V,dt", [(400, 7, 20001, "bf16"), (700, 3, 4097, "f32"), (500, 0, 33, "bf16")])
def test_lazy_and_eager_greedy_reads_agree(B, G, V, dt):
    """Greedy request claims (two CTAs per SM) read target rows one at a time
    up to the first draft that differs from its row's argmax.  Drafts are
    planted as the argmax of their target row with probability 0.8, so both
    early mismatches and full matches occur.  Lazy and eager reads agree bit
    for bit, and both with the oracle."""
    import numpy as np
    w = W.make_random(B, G, V, dt, seed=91 * B + G, gamma="ragged").to(DEV)
    assert route(w.target.dtype, B, G, V, greedy=True, sched=binding.SCHEDULE_STREAM) == \
        (binding.ROUTE_CLAIMS, 1)
    rng = np.random.default_rng(B)
    am = w.target[:, :G].float().argmax(dim=-1).to(torch.int32) if G > 0 else \
        torch.zeros((B, 0), dtype=torch.int32, device=DEV)
    keep = torch.as_tensor(rng.random((B, G)) < 0.8, device=DEV)
    other = torch.as_tensor(rng.integers(0, V, (B, G)), dtype=torch.int32, device=DEV)
    tokens = torch.where(keep, am, other).contiguous()
    lazy = _claims_greedy(w, tokens, True)
    eager = _claims_greedy(w, tokens, False)
    assert (lazy[0] == eager[0]).all() and (lazy[1] == eager[1]).all()
    ins = W.oracle_inputs(w)
    ref = oracle.greedy(ins["target"], tokens.cpu().numpy(), ins["gamma"], nthreads=NTHREADS)
    assert not compare_greedy(ref, lazy[0], lazy[1])
    if G > 0:
        n, g = lazy[1], w.gamma.cpu().numpy()
        assert (n < g).any() and ((n == g) & (g > 0)).any()
