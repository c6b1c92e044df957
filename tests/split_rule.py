"""The library's split plan, restated for the tests.

This is the product's documented partition rule (the decode path of
pa_attention: ranges of S = 512 * 2^j keys, j the smallest that leaves at most
128 ranges, so S depends on a row's own key count only), not part of the
attention definition: any partition folds back to the same fp64 attention.
The tests use it where the rule itself matters -- to cut KV-parallel owner
bounds on split edges, and to count the sequential accumulation steps that a
row's rounding-error bound charges for.
"""


def split_length(keys: int, base: int = 512, max_splits: int = 128) -> int:
    """Keys per split of a row with ``keys`` keys."""
    s = base
    while -(-keys // s) > max_splits:
        s *= 2
    return s


def split_starts(keys: int):
    """First key of every split of a row with ``keys`` keys."""
    s = split_length(keys)
    return list(range(0, keys, s))
