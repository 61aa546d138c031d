"""The prefix cache's host-side decisions, with a stand-in decoder (no GPU):
which cached prefix a prompt reuses, how many positions are copied, and
what is left to prefill."""
import torch

from invariant_deterministic_gb300.model import PrefixCache


class FakeDecoder:
    def __init__(self):
        self.calls = []

    def copy_prefix(self, src, dst, n):
        self.calls.append(("copy", src, dst, n))

    def prefill(self, seq, tokens, p0=0, chunk=0):
        self.calls.append(("prefill", seq, tokens.tolist(), p0))
        return torch.zeros(1)


def test_longest_registered_prefix():
    pc = PrefixCache(None)
    assert pc.longest([1, 2, 3]) == (None, 0)
    pc.insert([1, 2], slot=4)
    pc.insert([1, 2, 3, 4], slot=5)
    pc.insert([9], slot=6)
    assert pc.longest([1, 2, 3, 4, 5]) == (5, 4)
    assert pc.longest([1, 2, 3]) == (4, 2)      # [1, 2, 3, 4] is longer than the prompt
    assert pc.longest([1, 3]) == (None, 0)      # a prefix must match from the start
    assert pc.longest([9, 9]) == (6, 1)
    assert pc.longest([]) == (None, 0)


def test_prefill_copies_the_prefix_and_prefills_the_rest():
    dec = FakeDecoder()
    pc = PrefixCache(dec)
    pc.insert([7, 8, 9], slot=0)
    n, _ = pc.prefill(2, torch.tensor([7, 8, 9, 10, 11]))
    assert n == 3
    assert dec.calls == [("copy", 0, 2, 3), ("prefill", 2, [10, 11], 3)]


def test_a_whole_cached_prompt_recomputes_its_last_token():
    dec = FakeDecoder()
    pc = PrefixCache(dec)
    pc.insert([7, 8, 9], slot=0)
    n, _ = pc.prefill(1, torch.tensor([7, 8, 9]))
    assert n == 2                                   # the last row's hidden state is the output
    assert dec.calls == [("copy", 0, 1, 2), ("prefill", 1, [9], 2)]


def test_no_copy_onto_itself_and_nothing_cached():
    dec = FakeDecoder()
    pc = PrefixCache(dec)
    pc.insert([5, 6], slot=3)
    n, _ = pc.prefill(3, torch.tensor([5, 6, 7]))  # the prefix already sits in this slot
    assert n == 2 and dec.calls == [("prefill", 3, [7], 2)]
    dec.calls.clear()
    n, _ = pc.prefill(1, torch.tensor([1, 2]))
    assert n == 0 and dec.calls == [("prefill", 1, [1, 2], 0)]
