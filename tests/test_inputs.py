"""The seeded input recipe: the bits are a function of the seed alone, and the
logged SHA-256 over them identifies them."""
import torch

from exact_attention_blackwell_gb300 import inputs


def test_input_bits_and_hash_follow_the_seed():
    w = inputs.Workload("tiny", 1, 2, 2, 128, 64, False, 0)
    a, b = inputs.make_inputs(w), inputs.make_inputs(w)
    for n in ("q", "k", "v", "dO"):
        assert a[n].dtype == torch.bfloat16 and torch.equal(a[n].view(torch.int16), b[n].view(torch.int16))
    assert inputs.input_sha256(a) == inputs.input_sha256(b)
    other = inputs.make_inputs(inputs.Workload("tiny", 1, 2, 2, 128, 64, False, 1))
    assert inputs.input_sha256(other) != inputs.input_sha256(a)
    no_do = dict(a, dO=None)
    assert inputs.input_sha256(no_do) != inputs.input_sha256(a)
