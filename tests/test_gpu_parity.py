"""CUDA path vs the float64 oracle, through the C ABI (GPU).

With SV_PARITY_OUT set to a directory, the full-size workload tests write
their near-tie counts there (one JSON file per workload and mode)."""
import functools
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import softmax as scipy_softmax

import oracle
from parity import Report, compare_greedy, compare_sample, PROB_RTOL
from speculative_decoding_verification_62_gb300 import binding
from speculative_decoding_verification_62_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
NTHREADS = os.cpu_count() or 1


def run_gpu_sample(w, with_probs=True):
    v = binding.Verifier(w.B, w.G, w.V, DEV)
    p = torch.full((w.B, w.G), float("nan"), dtype=torch.float64, device=DEV) if with_probs else None
    q = torch.full_like(p, float("nan")) if with_probs else None
    v.sample(w.target, w.draft, w.draft_tokens, w.gamma, w.uniforms, w.temperature, p, q)
    torch.cuda.synchronize()
    st = binding.spec_verify_status(v.workspace)
    res = dict(out=v.out_tokens.cpu().numpy(), nacc=v.num_accepted.cpu().numpy(),
               p=None if p is None else p.cpu().numpy(), q=None if q is None else q.cpu().numpy())
    res["status"] = st
    res["ws_clean"] = bool(torch.count_nonzero(v.workspace[:counters_end(w.B)]) == 0)
    return res


def counters_end(B):
    """End of the header words (1 KiB), the two per-request arrival counters
    and the per-request decision records: all zero again after every call."""
    a256 = lambda n: (n + 255) // 256 * 256  # noqa: E731
    return 1024 + 2 * a256(4 * B) + a256(32 * B)


def check_sample_parity(w, requests=None):
    g = run_gpu_sample(w)
    assert g["status"] == 0, binding.status_names(g["status"])
    idx = np.arange(w.B) if requests is None else np.asarray(requests)
    ref = oracle.sample(**W.oracle_inputs(w, idx), nthreads=NTHREADS)
    rep = compare_sample(ref, g["out"][idx], g["nacc"][idx], w.gamma.cpu().numpy()[idx],
                         g["p"][idx], g["q"][idx])
    print(w.name, rep.summary())
    assert not rep.mismatches, rep.mismatches[:5]
    assert rep.max_prob_rel_err < PROB_RTOL
    return rep, g


def to_dev(w):
    return w.to(DEV)


SMALL = [
    (3, 2, 1, "bf16"), (4, 3, 7, "bf16"), (4, 3, 8, "f32"), (5, 2, 33, "bf16"),
    (6, 4, 4097, "bf16"), (6, 4, 4097, "f32"), (4, 3, 8192, "bf16"), (5, 3, 8193, "bf16"),
    (7, 5, 20000, "bf16"), (3, 7, 20001, "f32"), (9, 1, 65536, "bf16"),
]


@pytest.mark.parametrize("B,G,V,dt", SMALL)
def test_sample_small_ragged(B, G, V, dt):
    w = to_dev(W.make_random(B, G, V, dt, seed=B * 1000 + V, gamma="ragged",
                             temperature=[0.5 + 0.37 * i for i in range(B)], sigma_d=0.8))
    check_sample_parity(w)


@pytest.mark.parametrize("B,G,V,dt", SMALL)
def test_greedy_small_ragged(B, G, V, dt):
    w = to_dev(W.make_random(B, G, V, dt, seed=B * 1000 + V + 1, gamma="ragged"))
    # make some drafts match the argmax so acceptance runs deep
    am = w.target[:, :G].float().argmax(dim=2).to(torch.int32)
    keep = torch.rand(w.draft_tokens.shape, device=DEV) < 0.7
    tokens = torch.where(keep, am, w.draft_tokens)
    for b in range(B):
        tokens[b, int(w.gamma[b]):] = 0
    v = binding.Verifier(B, G, V, DEV)
    v.greedy(w.target, tokens.contiguous(), w.gamma)
    ref = oracle.greedy(W.logits_numpy(w.target), tokens.cpu().numpy(), w.gamma.cpu().numpy())
    bad = compare_greedy(ref, v.out_tokens.cpu().numpy(), v.num_accepted.cpu().numpy())
    assert not bad, bad[:5]
    assert binding.spec_verify_status(v.workspace) == 0


@functools.lru_cache(maxsize=1)
def full_size(name):
    """One standard workload on the device (drawn once per name and kept for
    the sampling and greedy tests of that name)."""
    return W.make(name, device=DEV)


def record(name, mode, w, payload):
    out = os.environ.get("SV_PARITY_OUT")
    if not out:
        return
    os.makedirs(out, exist_ok=True)
    route, csize = binding.spec_verify_route(w.target.dtype, w.B, w.G, w.V, greedy=mode == "greedy")
    payload = dict(workload=name, mode=mode, B=w.B, G=w.G, V=w.V, input_sha256=w.sha256(),
                   route=route, cluster_size=csize, **payload)
    with open(os.path.join(out, f"parity_{name}_{mode}.json"), "w") as f:
        json.dump(payload, f, indent=1)


@pytest.mark.parametrize("name", ["1", "2", "3", "4", "5a", "5b"])
def test_sample_full_size_configs(name):
    """Every request of each standard workload against the oracle."""
    w = full_size(name)
    rep, g = check_sample_parity(w)
    assert g["ws_clean"]
    record(name, "sample", w, rep.to_dict())


@pytest.mark.parametrize("name", ["2", "3", "4", "5a", "5b"])
def test_greedy_full_size_configs(name):
    """Every request, bit-exact; exact argmax ties are counted."""
    w = full_size(name)
    tokens = w.draft[:, :, :].float().argmax(dim=2).to(torch.int32)  # x = argmax of the draft
    for b in range(w.B):
        tokens[b, int(w.gamma[b]):] = 0
    tokens = tokens.contiguous()
    v = binding.Verifier(w.B, w.G, w.V, DEV)
    v.greedy(w.target, tokens, w.gamma)
    ref = oracle.greedy(W.logits_numpy(w.target), tokens.cpu().numpy(), w.gamma.cpu().numpy(),
                        nthreads=NTHREADS)
    bad = compare_greedy(ref, v.out_tokens.cpu().numpy(), v.num_accepted.cpu().numpy())
    assert not bad, bad[:5]
    g = w.gamma.cpu().numpy()
    ties = sum(int(ref["exact_tie"][b][:int(ref["num_accepted"][b]) + 1].sum()) for b in range(w.B))
    record(name, "greedy", w, dict(requests=w.B, rows_decided=int(sum(
        min(int(ref["num_accepted"][b]) + 1, int(g[b]) + 1) for b in range(w.B))),
        exact_argmax_ties=ties, mismatches=len(bad)))


def test_workspace_reuse_many_calls():
    """The kernels reset their counters: repeated calls on one workspace agree."""
    w = to_dev(W.make_random(16, 4, 30000, "bf16", seed=5, gamma="ragged"))
    v = binding.Verifier(w.B, w.G, w.V, DEV)
    v.sample(w.target, w.draft, w.draft_tokens, w.gamma, w.uniforms, w.temperature)
    first = (v.out_tokens.clone(), v.num_accepted.clone())
    for _ in range(5):
        v.sample(w.target, w.draft, w.draft_tokens, w.gamma, w.uniforms, w.temperature)
        v.greedy(w.target, w.draft_tokens, w.gamma)
        v.sample(w.target, w.draft, w.draft_tokens, w.gamma, w.uniforms, w.temperature)
        assert torch.equal(v.out_tokens, first[0]) and torch.equal(v.num_accepted, first[1])
    assert not v.workspace[:counters_end(w.B)].cpu().numpy().any()


def test_q_equals_p_accepts_all_gpu():
    w = to_dev(W.make_random(32, 5, 5000, "bf16", seed=8))
    w.draft.copy_(w.target[:, :5])
    u = w.uniforms.clone()
    u[:, :5] = torch.where(torch.rand_like(u[:, :5]) < 0.3, torch.full_like(u[:, :5], 0.99999994),
                           u[:, :5])
    w.uniforms.copy_(u)
    g = run_gpu_sample(w)
    assert np.all(g["nacc"] == 5)
    assert np.array_equal(g["out"][:, :5], w.draft_tokens.cpu().numpy())


def test_disjoint_supports_reject_at_zero_gpu():
    B, G, V = 64, 3, 1000
    t = torch.full((B, G + 1, V), -1.0e4, device=DEV)
    d = torch.full((B, G, V), -1.0e4, device=DEV)
    t[:, :, :500] = torch.randn((B, G + 1, 500), device=DEV)
    d[:, :, 500:] = torch.randn((B, G, 500), device=DEV)
    w = W.Workload("disjoint", t.to(torch.bfloat16).contiguous(), d.to(torch.bfloat16).contiguous(),
                   torch.randint(500, 1000, (B, G), device=DEV, dtype=torch.int32),
                   torch.full((B,), G, dtype=torch.int32, device=DEV),
                   torch.rand((B, G + 1), device=DEV), torch.ones(B, device=DEV))
    rep, g = check_sample_parity(w)
    assert np.all(g["nacc"] == 0) and np.all(g["out"][:, 0] < 500)


def test_masked_logits_gpu():
    w = to_dev(W.make_random(12, 3, 9000, "bf16", seed=9, gamma="ragged"))
    mask = torch.rand(w.target.shape, device=DEV) < 0.3
    w.target.masked_fill_(mask, float("-inf"))
    w.draft.masked_fill_(mask[:, :3], float("-inf"))
    w.draft.masked_fill_(torch.rand(w.draft.shape, device=DEV) < 0.1, float("-inf"))
    rep, g = check_sample_parity(w)
    for b in range(w.B):  # a token masked in the target row is never drawn
        k = g["nacc"][b]
        assert not bool(mask[b, k, g["out"][b, k]])


def test_inverse_cdf_exact_boundaries_gpu():
    cases = [(0.0, 0), (0.2499, 0), (0.25, 1), (0.4999999, 1), (0.5, 2), (0.75, 3),
             (0.99999994, 3)]
    n = len(cases)
    t = torch.zeros((n, 1, 4), dtype=torch.bfloat16, device=DEV)
    u = torch.tensor([[c[0]] for c in cases], dtype=torch.float32, device=DEV)
    v = binding.Verifier(n, 0, 4, DEV)
    v.sample(t, None, None, torch.zeros(n, dtype=torch.int32, device=DEV), u,
             torch.ones(n, device=DEV))
    assert v.out_tokens[:, 0].cpu().tolist() == [c[1] for c in cases]
    assert v.num_accepted.cpu().tolist() == [0] * n


def test_accept_is_strict_gpu():
    t = torch.zeros((2, 2, 4), dtype=torch.float32, device=DEV)
    d = torch.tensor([[[0.0, 0.0, -math.inf, -math.inf]]] * 2, device=DEV)
    u = torch.tensor([[0.5, 0.3], [0.49999997, 0.3]], device=DEV)
    v = binding.Verifier(2, 1, 4, DEV)
    p = torch.empty((2, 1), dtype=torch.float64, device=DEV)
    q = torch.empty_like(p)
    v.sample(t, d.contiguous(), torch.zeros((2, 1), dtype=torch.int32, device=DEV),
             torch.ones(2, dtype=torch.int32, device=DEV), u, torch.ones(2, device=DEV), p, q)
    assert v.num_accepted.cpu().tolist() == [0, 1]
    assert p.cpu().tolist() == [[0.25], [0.25]] and q.cpu().tolist() == [[0.5], [0.5]]


def test_expected_tokens_closed_form_gpu():
    """Mean emitted tokens over 1e5 requests matches (1 - a^(g+1))/(1 - a)."""
    B, G = 100_000, 3
    t = torch.log(torch.tensor([0.8, 0.2])).float()
    d = torch.log(torch.tensor([0.5, 0.5])).float()
    p = scipy_softmax(t.double().numpy())
    q = scipy_softmax(d.double().numpy())
    alpha = float(np.minimum(p, q).sum())
    gen = torch.Generator(device=DEV).manual_seed(11)
    tgt = t.to(DEV).view(1, 1, 2).expand(B, G + 1, 2).contiguous()
    dft = d.to(DEV).view(1, 1, 2).expand(B, G, 2).contiguous()
    x = (torch.rand((B, G), generator=gen, device=DEV) >= float(q[0])).to(torch.int32)
    u = torch.rand((B, G + 1), generator=gen, device=DEV)
    v = binding.Verifier(B, G, 2, DEV)
    v.sample(tgt, dft, x, torch.full((B,), G, dtype=torch.int32, device=DEV), u,
             torch.ones(B, device=DEV))
    n = v.num_accepted.double() + 1
    mean, se = float(n.mean()), float(n.std()) / math.sqrt(B)
    expect = (1 - alpha ** (G + 1)) / (1 - alpha)
    assert abs(mean - expect) < 5 * se, (mean, expect, se)


def test_emitted_law_equals_p_gpu():
    """First emitted token over 200k identical requests follows p (V = 20,
    gamma = 5, q from 0.7 x the target logits, as in the theory page's check)."""
    B, G, V = 200_000, 5, 20
    rng = np.random.default_rng(42)
    logits = (rng.normal(0, 1, V) * 2.0).astype(np.float32)
    dl = (0.7 * logits).astype(np.float32)
    p = scipy_softmax(logits.astype(np.float64))
    q = scipy_softmax(dl.astype(np.float64))
    gen = torch.Generator(device=DEV).manual_seed(12)
    tgt = torch.from_numpy(logits).to(DEV).view(1, 1, V).expand(B, G + 1, V).contiguous()
    dft = torch.from_numpy(dl).to(DEV).view(1, 1, V).expand(B, G, V).contiguous()
    x = torch.multinomial(torch.from_numpy(q).float().to(DEV).expand(B * G, V), 1,
                          generator=gen).view(B, G).to(torch.int32).contiguous()
    u = torch.rand((B, G + 1), generator=gen, device=DEV)
    v = binding.Verifier(B, G, V, DEV)
    v.sample(tgt, dft, x, torch.full((B,), G, dtype=torch.int32, device=DEV), u,
             torch.ones(B, device=DEV))
    first = v.out_tokens[:, 0].cpu().numpy()
    freq = np.bincount(first, minlength=V) / B
    assert np.all(np.abs(freq - p) < 5 * np.sqrt(p * (1 - p) / B) + 1e-9)


def test_status_flags_on_invalid_device_values():
    """Out-of-range device values are clamped in the kernels and reported."""
    w = to_dev(W.make_random(6, 3, 3000, "bf16", seed=13))
    w.gamma[0] = 9
    w.gamma[1] = -2
    w.draft_tokens[2, 0] = 3000
    w.uniforms[3, 0] = 1.5
    w.temperature[4] = -1.0
    v = binding.Verifier(w.B, w.G, w.V, DEV)
    v.sample(w.target, w.draft, w.draft_tokens, w.gamma, w.uniforms, w.temperature)
    st = binding.spec_verify_status(v.workspace)
    for bit in ("BAD_GAMMA", "BAD_TOKEN", "BAD_UNIFORM", "BAD_TEMPERATURE"):
        assert bit in binding.status_names(st), binding.status_names(st)
    nacc = v.num_accepted.cpu().numpy()
    assert 0 <= nacc[0] <= 3 and nacc[1] == 0
    assert binding.spec_verify_status(v.workspace) == 0  # read clears


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_zero_temperature_requests_are_greedy_in_a_sampling_call(dt):
    """T_b = 0 verifies request b by argmax matching inside the sampling launch."""
    B, G, V = 12, 4, 20001
    w = to_dev(W.make_random(B, G, V, dt, seed=77, gamma="ragged",
                             temperature=[0.6 + 0.1 * i for i in range(B)]))
    am = w.target[:, :G].float().argmax(dim=2).to(torch.int32)
    for b in range(0, B, 3):
        w.temperature[b] = 0.0
        w.draft_tokens[b] = am[b]
        if b % 2:
            w.draft_tokens[b, 1] = (am[b, 1] + 1) % V   # a mismatch at position 1
        w.draft_tokens[b, int(w.gamma[b]):] = 0
    rep, g = check_sample_parity(w)
    assert g["ws_clean"]
    ref_g = oracle.greedy(W.logits_numpy(w.target), w.draft_tokens.cpu().numpy(),
                          w.gamma.cpu().numpy())
    for b in range(0, B, 3):
        assert (g["out"][b] == ref_g["out_tokens"][b]).all()
        assert g["nacc"][b] == ref_g["num_accepted"][b]
        assert np.isnan(g["p"][b]).all() and np.isnan(g["q"][b]).all()


@pytest.mark.parametrize("V,dt", [(128256, "bf16"), (32000, "f32"), (4097, "bf16"), (1, "f32")])
def test_draft_sampler_matches_oracle(V, dt):
    """spec_verify_draw: one token per row from softmax(z / T) by inverse CDF."""
    B = 48
    w = W.make_random(B, 0, V, dt, seed=V + 3, temperature=[0.5 + 0.05 * i for i in range(B)])
    w.temperature[::7] = 0.0                     # argmax rows
    w = to_dev(w)
    logits = w.target[:, 0].contiguous()
    u = w.uniforms[:, 0].contiguous()
    tokens = torch.full((B,), -5, dtype=torch.int32, device=DEV)
    ws = binding.make_workspace(B, 0, V)
    binding.spec_verify_draw(logits, u, w.temperature, tokens, ws)
    torch.cuda.synchronize()
    assert binding.spec_verify_status(ws) == 0
    ref = oracle.sample(**W.oracle_inputs(w), nthreads=NTHREADS)
    rep = compare_sample(ref, tokens.cpu().numpy()[:, None], np.zeros(B, np.int32),
                         np.zeros(B, np.int32))
    print(w.name, rep.summary())
    assert not rep.mismatches, rep.mismatches[:5]
    tk = tokens.cpu().numpy()
    am = logits.float().argmax(dim=1).cpu().numpy()
    z = (w.temperature.cpu().numpy() == 0)
    assert (tk[z] == am[z]).all()
