"""Cluster schedule (small batches) vs the persistent grid and the oracle (GPU).

Both schedules compute every value with the same arithmetic, so their
outputs must agree bit for bit; the cluster results are also compared with the
float64 oracle."""
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


def sample_both(w, probs=True, packed=False):
    """(cluster-schedule result, persistent result), each (out, nacc, p, q)."""
    res = []
    for sched in (binding.SCHEDULE_AUTO, binding.SCHEDULE_PERSISTENT):
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


def same(a, b):
    (oa, na, pa, qa), (ob, nb, pb, qb) = a, b
    assert (oa == ob).all() and (na == nb).all()
    for x, y in ((pa, pb), (qa, qb)):
        if x is None:
            continue
        nan = torch.isnan(y)
        assert torch.equal(torch.isnan(x), nan)
        assert torch.equal(x[~nan], y[~nan])


def against_oracle(w, res):
    out, nacc, p, q = res
    ref = oracle.sample(**W.oracle_inputs(w), nthreads=NTHREADS)
    rep = compare_sample(ref, out, nacc, w.gamma.cpu().numpy(),
                         None if p is None else p.numpy(), None if q is None else q.numpy())
    print(w.name, rep.summary())
    assert not rep.mismatches, rep.mismatches[:5]
    assert rep.max_prob_rel_err < PROB_RTOL


def test_small_batches_take_the_cluster_schedule():
    """One wave of clusters whose warps hold one unit each of a request's work
    (a unit: an 8 KB target chunk and the draft chunk of the same position)."""
    bf, f32 = torch.bfloat16, torch.float32
    for dt in (bf, f32):
        assert binding.spec_verify_cluster_size(dt, 1, 4, 32000) > 0
        assert binding.spec_verify_cluster_size(dt, 8, 3, 32000) > 0
        assert binding.spec_verify_cluster_size(dt, 512, 3, 128256) == 0
    assert binding.spec_verify_cluster_size(bf, 8, 3, 128256) > 0
    assert binding.spec_verify_cluster_size(bf, 8, 3, 128256, greedy=True) > 0
    # too many units per request for one cluster: the persistent grid
    assert binding.spec_verify_cluster_size(f32, 2, 3, 128256) == 0
    assert binding.spec_verify_cluster_size(bf, 2, 31, 128256) == 0
    prev = binding.spec_verify_set_schedule(binding.SCHEDULE_PERSISTENT)
    try:
        assert binding.spec_verify_cluster_size(torch.bfloat16, 8, 3, 128256) == 0
    finally:
        binding.spec_verify_set_schedule(prev)


CASES = [(8, 3, 128256, "bf16"), (5, 4, 20001, "bf16"), (3, 2, 4097, "f32"), (1, 4, 32000, "f32"),
         (6, 7, 8193, "bf16"), (4, 3, 1, "bf16"), (7, 4, 152064, "bf16"), (2, 3, 32000, "f32")]


@pytest.mark.parametrize("B,G,V,dt", CASES)
def test_cluster_sample_matches_persistent_and_oracle(B, G, V, dt):
    temps = [0.6 + 0.15 * i for i in range(B)]
    w = W.make_random(B, G, V, dt, seed=B * 101 + V, gamma="ragged", temperature=temps).to(DEV)
    assert binding.spec_verify_cluster_size(w.target.dtype, B, G, V) > 0
    a, b = sample_both(w)
    same(a, b)
    against_oracle(w, a)


def test_cluster_full_size_config2():
    w = W.make("2", device=DEV)
    assert binding.spec_verify_cluster_size(w.target.dtype, w.B, w.G, w.V) > 0
    a, b = sample_both(w)
    same(a, b)
    against_oracle(w, a)


def test_cluster_zero_temperature_and_packed():
    B, G, V = 6, 4, 30001
    temps = [0.0, 0.8, 1.3, 0.0, 0.5, 1.0]
    w = W.make_random(B, G, V, "bf16", seed=5, gamma=[4, 0, 2, 3, 4, 1], temperature=temps).to(DEV)
    a, b = sample_both(w)
    same(a, b)
    against_oracle(w, a)
    c, d = sample_both(w, packed=True)
    same(c, d)
    same(a, c)


def test_cluster_rejections_and_bonus_both_occur():
    """Sharp rows with far-off drafts reject; identical rows accept (bonus)."""
    B, G, V = 8, 3, 50000
    w = W.make_random(B, G, V, "bf16", seed=9, sigma_t=4.0, sigma_d=3.0).to(DEV)
    w.draft[::2] = w.target[::2, :G]  # even requests: q == p, every draft accepted
    a, b = sample_both(w)
    same(a, b)
    nacc = a[1]
    assert (nacc[::2] == G).all() and (nacc[1::2] < G).any()
    against_oracle(w, a)


@pytest.mark.parametrize("B,G,V,dt", [(8, 3, 128256, "bf16"), (5, 6, 20001, "f32"), (2, 0, 7, "bf16")])
def test_cluster_greedy_matches_persistent_and_oracle(B, G, V, dt):
    w = W.make_random(B, G, V, dt, seed=B + V, gamma="ragged").to(DEV)
    if G:
        am = w.target[:, :G].float().argmax(dim=2).to(torch.int32)
        keep = torch.rand(w.draft_tokens.shape, device=DEV) < 0.7
        w.draft_tokens = torch.where(keep, am, w.draft_tokens).contiguous()
        for b in range(B):
            w.draft_tokens[b, int(w.gamma[b]):] = 0
    outs = []
    for sched in (binding.SCHEDULE_AUTO, binding.SCHEDULE_PERSISTENT):
        prev = binding.spec_verify_set_schedule(sched)
        try:
            v = binding.Verifier(B, G, V, DEV)
            v.greedy(w.target, w.draft_tokens, w.gamma)
            torch.cuda.synchronize()
            assert binding.spec_verify_status(v.workspace) == 0
            outs.append((v.out_tokens.cpu().numpy(), v.num_accepted.cpu().numpy()))
        finally:
            binding.spec_verify_set_schedule(prev)
    assert (outs[0][0] == outs[1][0]).all() and (outs[0][1] == outs[1][1]).all()
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
    for sched in (binding.SCHEDULE_AUTO, binding.SCHEDULE_PERSISTENT):
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
    assert torch.equal(toks[0], toks[1])


def test_cluster_status_flags_and_reuse():
    """Invalid device values are flagged on the cluster path too; repeated
    calls on one workspace keep it usable."""
    B, G, V = 4, 3, 5000
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


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_vanished_residual_falls_back_to_p_on_both_schedules(dt):
    """A clear rejection whose residual mass is below the fixed-point
    resolution: the drafted token x has q(x) = 2 p(x) with p(x) ~ e^-40 and
    the target and draft rows agree elsewhere, so u = 0.9 rejects (ratio 1/2)
    while sum max(0, p - q) ~ p(x) rounds to 0 in units of 2^-39.  Both
    schedules then draw from p_k; their tokens must agree, and the token must
    have p > 0.  (The float64 oracle's residual is pure cancellation noise
    here, so it is not the reference for this case.)"""
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
    res = sample_both(w, probs=False)
    assert binding.spec_verify_cluster_size(w.target.dtype, B, G, V) > 0
    same(res[0], res[1])
    out, nacc = res[0][0], res[0][1]
    assert (nacc == 0).all()
    p = torch.softmax(w.target[:, 0].double(), dim=1).cpu()
    for b in range(B):
        assert 0 <= out[b, 0] < V and out[b, 0] != x and p[b, out[b, 0]] > 0
        assert out[b, 1] == -1


def test_batch_at_the_cluster_wave_limit():
    """The largest batch that fits one wave of clusters runs on the cluster
    schedule, one more request runs on the persistent grid; both match the
    oracle."""
    G, V = 2, 32000
    limit = max(B for B in range(1, 65)
                if binding.spec_verify_cluster_size(torch.bfloat16, B, G, V) > 0)
    assert binding.spec_verify_cluster_size(torch.bfloat16, limit + 1, G, V) == 0
    for B in (limit, limit + 1):
        w = W.make_random(B, G, V, "bf16", seed=B, gamma="ragged",
                          temperature=[0.7 + 0.02 * i for i in range(B)]).to(DEV)
        a, b = sample_both(w)
        same(a, b)
        against_oracle(w, a)
