"""The seeded input generator: determinism, shapes and the draft-token law (CPU)."""
import numpy as np
import torch
from scipy.special import softmax as scipy_softmax

from speculative_decoding_verification_62_gb300 import workloads as W


def test_deterministic_and_shaped():
    a = W.make_random(5, 3, 100, "bf16", seed=3, gamma="ragged", temperature=[0.5, 1, 1.5, 2, 1])
    b = W.make_random(5, 3, 100, "bf16", seed=3, gamma="ragged", temperature=[0.5, 1, 1.5, 2, 1])
    for k in ("target", "draft", "draft_tokens", "gamma", "uniforms", "temperature"):
        assert torch.equal(getattr(a, k), getattr(b, k))
    assert a.target.shape == (5, 4, 100) and a.draft.shape == (5, 3, 100)
    assert a.target.dtype == torch.bfloat16
    assert a.draft_tokens.dtype == torch.int32 and a.gamma.dtype == torch.int32
    assert torch.all((a.uniforms >= 0) & (a.uniforms < 1))
    assert torch.all((a.gamma >= 0) & (a.gamma <= 3))
    assert torch.all((a.draft_tokens >= 0) & (a.draft_tokens < 100))


def test_config1_shapes():
    w = W.make("1")
    assert (w.B, w.G, w.V) == (1, 4, 32000) and w.target.dtype == torch.float32
    assert w.bytes_min() > 4 * 32000 * 9


def test_gumbel_max_draws_follow_q():
    """x ~ softmax(d/T): frequencies over 200k rows match scipy's softmax."""
    g = torch.Generator().manual_seed(0)
    d = torch.tensor([0.0, 1.0, -0.5, 2.0])
    n = 200_000
    rows = d.view(1, 1, 4).expand(n, 1, 4).contiguous()
    T = torch.full((n,), 0.8)
    x = W.gumbel_max_tokens(rows, T, g).view(-1).numpy()
    freq = np.bincount(x, minlength=4) / n
    q = scipy_softmax(d.double().numpy() / np.float64(np.float32(0.8)))
    assert np.all(np.abs(freq - q) < 5 * np.sqrt(q * (1 - q) / n))


def test_oracle_inputs_roundtrip_bf16_bits():
    w = W.make_random(2, 2, 16, "bf16", seed=1)
    o = W.oracle_inputs(w)
    assert o["target"].dtype == np.uint16
    back = torch.from_numpy(o["target"].view(np.int16)).view(torch.bfloat16)
    assert torch.equal(back, w.target)


def test_input_digest_names_the_bytes():
    """The bench reports the inputs' SHA-256: equal seeds give equal digests,
    and any change of the bytes changes it."""
    a = W.make_random(3, 2, 50, "bf16", seed=5)
    b = W.make_random(3, 2, 50, "bf16", seed=5)
    c = W.make_random(3, 2, 50, "bf16", seed=6)
    assert a.sha256() == b.sha256() and len(a.sha256()) == 64
    assert a.sha256() != c.sha256()
    b.uniforms[0, 0] = 0.5 if float(b.uniforms[0, 0]) != 0.5 else 0.25
    assert a.sha256() != b.sha256()
    assert W.make_random(1, 0, 7, "f32", seed=1).sha256() == W.make_random(1, 0, 7, "f32", seed=1).sha256()


def test_bytes_needed_counts_rows_up_to_the_first_rejection():
    """Lazily read, a sampled request needs target and draft rows 0..k (k the
    first rejected position) and the bonus row only after a full acceptance;
    a greedy request (T == 0) needs target rows 0..k; eagerly, every row.
    Rows counted by hand for gamma = (3, 3, 3, 2, 0, 3)."""
    w = W.make_random(6, 3, 16, "bf16", seed=5, gamma=[3, 3, 3, 2, 0, 3],
                      temperature=[1.0, 1.0, 1.0, 1.0, 1.0, 0.0])
    k = torch.tensor([0, 1, 3, 2, 0, 1], dtype=torch.int32)
    small = w.bytes_min("sample") - (2 * 14 + 6) * 16 * 2  # the same small terms
    # rows: k=0 -> 2; k=1 -> 4; k=3=gamma -> 6 + 1; k=2=gamma(2) -> 4 + 1;
    # gamma 0 -> the bonus row; greedy with k = 1 -> target rows 0 and 1
    rows = 2 + 4 + 7 + 5 + 1 + 2
    assert w.bytes_needed("sample", k, lazy=True, ctas=1) == rows * 16 * 2 + small
    assert w.bytes_needed("sample", k, lazy=False, ctas=1) == w.bytes_min("sample")
    assert w.bytes_needed("greedy", k, lazy=False, ctas=1) == w.bytes_min("greedy")
    # greedy, lazily: target rows 0..k
    small_g = w.bytes_min("greedy") - (14 + 6) * 16 * 2
    assert w.bytes_needed("greedy", k, lazy=True, ctas=1) == (1 + 2 + 4 + 3 + 1 + 2) * 16 * 2 + small_g
    # fewer than two requests per CTA: sampled requests read whole (7, 7, 7,
    # 5, 1 rows), the greedy one still up to its first mismatch (2 rows)
    assert w.bytes_needed("sample", k, lazy=True, ctas=4) == (7 + 7 + 7 + 5 + 1 + 2) * 16 * 2 + small
