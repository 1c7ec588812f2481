"""A bounded wait that runs out ends the call with SV_STATUS_TIMEOUT instead
of hanging (GPU).

Failure is made on the host, never by a fault: the persistent grid's warps
that claim residual work in a queue slot past the last rejection wait until
either the slot is published or every request is decided (the workspace's
decision count reaches B).  Pre-setting that count, an in-bounds word of the
workspace, to a value it can never come back from keeps the second condition
false, so those warps wait for their limit, lowered here to 20 ms, set the
TIMEOUT bit and stop.  The call must return promptly with the bit set; after
the workspace is zero-filled again the next call is correct."""
import time

import numpy as np
import pytest
import torch

import oracle
from parity import compare_sample
from speculative_decoding_verification_62_gb300 import binding
from speculative_decoding_verification_62_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
DEC_COUNT_OFFSET = 640  # byte offset of the decision count in the workspace header


def test_queue_wait_runs_out_and_sets_timeout():
    B, G, V = 64, 2, 4096
    w = W.make_random(B, G, V, "bf16", seed=71)
    w.draft[0::2] = w.target[0::2, :G]  # q == p: every draft accepted, no queue slot
    w = w.to(DEV)
    prev_sched = binding.spec_verify_set_schedule(binding.SCHEDULE_PERSISTENT)
    prev_wait = binding.spec_verify_set_wait_limit(20_000_000)
    try:
        v = binding.Verifier(B, G, V, DEV)
        v.sample(w.target, w.draft, w.draft_tokens, w.gamma, w.uniforms, w.temperature)
        torch.cuda.synchronize()
        assert binding.spec_verify_status(v.workspace) == 0
        good = (v.out_tokens.clone(), v.num_accepted.clone())
        assert int((v.num_accepted[0::2] == G).sum()) == B // 2

        v.workspace.view(torch.int32)[DEC_COUNT_OFFSET // 4] = 1 << 30
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        v.sample(w.target, w.draft, w.draft_tokens, w.gamma, w.uniforms, w.temperature)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        st = binding.spec_verify_status(v.workspace)
        assert "TIMEOUT" in binding.status_names(st), binding.status_names(st)
        assert elapsed < 1.5, elapsed  # well under the 2 s default limit
        # the last CTA out still reset the header counters
        assert int(v.workspace.view(torch.int32)[DEC_COUNT_OFFSET // 4]) == 0

        v.workspace.zero_()
        v.sample(w.target, w.draft, w.draft_tokens, w.gamma, w.uniforms, w.temperature)
        torch.cuda.synchronize()
        assert binding.spec_verify_status(v.workspace) == 0
        assert torch.equal(v.out_tokens, good[0]) and torch.equal(v.num_accepted, good[1])
    finally:
        binding.spec_verify_set_wait_limit(prev_wait)
        binding.spec_verify_set_schedule(prev_sched)
    ref = oracle.sample(**W.oracle_inputs(w))
    rep = compare_sample(ref, good[0].cpu().numpy(), good[1].cpu().numpy(), w.gamma.cpu().numpy())
    assert not rep.mismatches, rep.mismatches
    _ = np
