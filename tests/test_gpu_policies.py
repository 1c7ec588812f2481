"""The draft-length policies fed by the GPU verify step's outputs (closed loop)."""
import numpy as np
import pytest
import torch

from speculative_decoding_verification_62_gb300 import binding
from speculative_decoding_verification_62_gb300 import policies as pol

pytestmark = pytest.mark.gpu
DEV = "cuda"


def verify_two_token(B, G, seed):
    """p = (0.8, 0.2), q = (0.5, 0.5) at every position: acceptance alpha = 0.7."""
    t = torch.log(torch.tensor([0.8, 0.2])).float()
    d = torch.log(torch.tensor([0.5, 0.5])).float()
    gen = torch.Generator(device=DEV).manual_seed(seed)
    tgt = t.to(DEV).view(1, 1, 2).expand(B, G + 1, 2).contiguous()
    dft = d.to(DEV).view(1, 1, 2).expand(B, G, 2).contiguous()
    x = (torch.rand((B, G), generator=gen, device=DEV) >= 0.5).to(torch.int32)
    u = torch.rand((B, G + 1), generator=gen, device=DEV)
    v = binding.Verifier(B, G, 2, DEV)
    gamma = torch.full((B,), G, dtype=torch.int32, device=DEV)
    v.sample(tgt, dft, x, gamma, u, torch.ones(B, device=DEV))
    return gamma.cpu().numpy(), v.num_accepted.cpu().numpy()


def test_estimator_recovers_alpha_from_gpu_outputs():
    est = pol.AcceptanceEstimator()
    for seed in range(4):
        g, k = verify_two_token(20_000, 4, seed)
        est.update(g, k)
    assert abs(est.alpha - 0.7) < 0.01
    assert abs(pol.optimal_gamma(est.alpha, 0.1) - pol.optimal_gamma(0.7, 0.1)) <= 1


def test_policies_in_a_closed_loop():
    ema = pol.AcceptLengthEMA(weight=0.5)
    table = pol.BatchSizeTable.docs_example()
    steps = ema.steps(4)
    for seed in range(5):
        g, k = verify_two_token(4, steps, 100 + seed)
        ema.observe(4, k)
        steps = ema.steps(4)
        assert 1 <= steps <= 7
    assert table(4) == 3
    rate = pol.acceptance_rate(g, k)
    assert 0.0 <= rate <= 1.0
