"""Host check of the 4096-point NTT kernels' shared-memory placement
(`Swz4096` in ntt_core.cuh), restated here: element a = 256 hi + 16 mid + lo
sits at 256 hi + 16 (mid ^ (hi & 1)) + (lo ^ mid).  The placement must be a
bijection of the row, the kernels' per-thread bases must give the same
positions, and every access pattern of the three radix-16 rounds must hit 32
distinct banks per warp (words, 32 banks)."""


def place(a):
    hi, mid, lo = a >> 8, (a >> 4) & 15, a & 15
    return (hi << 8) | ((mid ^ (hi & 1)) << 4) | (lo ^ mid)


def bases(t):
    """The kernel's per-thread bases (Swz4096's constructor)."""
    hi, lo = t >> 4, t & 15
    e0 = (hi << 4) | (lo ^ hi)
    e1 = ((hi ^ 1) << 4) | (lo ^ hi)
    b1 = (hi << 8) | ((hi & 1) << 4) | lo
    b2 = (hi << 8) | ((lo ^ (hi & 1)) << 4) | lo
    return e0, e1, b1, b2


PATTERNS = {
    "col": lambda t, i: t + 256 * i,                          # round 0 forward, round 2 inverse
    "mid": lambda t, i: 256 * (t >> 4) + (t & 15) + 16 * i,   # the middle round
    "row": lambda t, i: 16 * t + i,                           # round 2 forward, round 0 inverse
}


def test_placement_is_a_bijection():
    assert sorted(place(a) for a in range(4096)) == list(range(4096))


def test_thread_bases_give_the_placement():
    for t in range(256):
        e0, e1, b1, b2 = bases(t)
        for i in range(16):
            assert (e1 if i & 1 else e0) + 256 * i == place(PATTERNS["col"](t, i))
            assert b1 ^ (17 * i) == place(PATTERNS["mid"](t, i))
            assert b2 ^ i == place(PATTERNS["row"](t, i))


def test_every_round_is_free_of_bank_conflicts():
    for name, f in PATTERNS.items():
        for warp in range(8):
            for i in range(16):
                banks = {place(f(t, i)) % 32 for t in range(32 * warp, 32 * warp + 32)}
                assert len(banks) == 32, (name, warp, i)


def test_natural_placement_has_the_conflicts_it_replaced():
    """Without the swizzle the middle round is a 2-way and the row pattern a
    16-way bank conflict (word accesses)."""
    worst = {}
    for name, f in PATTERNS.items():
        worst[name] = max(32 // len({f(t, i) % 32 for t in range(32)}) for i in range(16))
    assert worst == {"col": 1, "mid": 2, "row": 16}
