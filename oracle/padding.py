"""Vocabulary padding rule. Test infrastructure.

[p1] §3.4, "Vocabulary padding for efficiency", and [p5] §3.4: each of the t
vocabulary shards should hold a multiple of 128 rows, so the vocabulary is
rounded up to the next multiple of 128 * t (GPT-2: 50,257 -> 51,200 at t = 8,
943 padding rows that no token uses).
"""


def pad_vocab(v: int, t: int, multiple: int = 128) -> int:
    """Smallest multiple of multiple * t that is >= v."""
    if v < 0 or t < 1 or multiple < 1:
        raise ValueError("pad_vocab: need v >= 0, t >= 1, multiple >= 1")
    q = multiple * t
    return ((v + q - 1) // q) * q
