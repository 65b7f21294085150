"""Shared-memory bank conflicts as the page "03_shared_memory_sync_reduction.py",
demo 1 (bank conflicts), describes them, and the page "simt_lab.py"
(`Block._shared_access`) counts them.

TEST INFRASTRUCTURE, NOT PRODUCT CODE (see ``oracle/__init__.py``).

Shared memory is split into 32 banks; 4-byte word k lives in bank k mod 32
and each bank serves one word per cycle.  A warp's access takes as many
rounds ("wavefronts") as the largest number of *distinct* words any one bank
is asked for; threads reading the same word share it (broadcast).
"""
from __future__ import annotations

N_BANKS = 32

# Demo 1's access patterns, by the index each thread tid of one warp reads
# (the array holds 32 * 33 words and the index is taken modulo that size).
ARRAY_WORDS = 32 * 33
PATTERNS = (
    ("stride 1", lambda t: t),
    ("stride 2", lambda t: 2 * t),
    ("stride 4", lambda t: 4 * t),
    ("stride 8", lambda t: 8 * t),
    ("stride 16", lambda t: 16 * t),
    ("stride 32 (a column of a 32x32 tile)", lambda t: 32 * t),
    ("stride 33 (a column of a 32x33 padded tile)", lambda t: 33 * t),
    ("stride 3 (odd)", lambda t: 3 * t),
    ("broadcast (one word)", lambda t: 0 * t),
    ("pairs share a word (tid // 2)", lambda t: t // 2),
)


def indices(pattern: int, warp: int = 32) -> list[int]:
    fn = PATTERNS[pattern][1]
    return [fn(t) % ARRAY_WORDS for t in range(warp)]


def wavefronts(words: list[int], n_banks: int = N_BANKS) -> int:
    """Rounds one warp-wide access to these 4-byte word indices takes."""
    distinct_per_bank: dict[int, set[int]] = {}
    for w in words:
        distinct_per_bank.setdefault(w % n_banks, set()).add(w)
    return max((len(v) for v in distinct_per_bank.values()), default=0)
