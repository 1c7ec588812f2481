"""Packing a padded workload (CPU): pure re-layout, checked element by element."""
import torch

from speculative_decoding_verification_62_gb300 import workloads as W


def test_pack_layout():
    w = W.make_random(5, 3, 17, "f32", seed=4, gamma=[0, 3, 1, 2, 0])
    p = W.pack(w)
    assert p.cu_draft.tolist() == [0, 0, 3, 4, 6, 6]
    assert p.target.shape == (6 + 5, 17) and p.draft.shape == (6, 17)
    rows = [(b, i) for b in range(5) for i in range(int(w.gamma[b]) + 1)]
    for r, (b, i) in enumerate(rows):
        assert torch.equal(p.target[r], w.target[b, i])
        u = w.uniforms[b, i] if i < int(w.gamma[b]) else w.uniforms[b, w.G]
        assert p.uniforms[r] == u
    drows = [(b, i) for b in range(5) for i in range(int(w.gamma[b]))]
    for r, (b, i) in enumerate(drows):
        assert torch.equal(p.draft[r], w.draft[b, i])
        assert p.draft_tokens[r] == w.draft_tokens[b, i]
    back = W.unpack_per_draft(p.draft_tokens.double(), p.cu_draft, w.G, fill=-1.0)
    for b in range(5):
        g = int(w.gamma[b])
        assert back[b, :g].tolist() == w.draft_tokens[b, :g].double().tolist()
        assert (back[b, g:] == -1).all()


def test_pack_without_drafts():
    w = W.make_random(3, 2, 9, "bf16", seed=5, gamma=[0, 0, 0])
    p = W.pack(w)
    assert p.total == 0 and p.draft.shape == (0, 9) and p.target.shape == (3, 9)
