"""The code maps, decoded bit pattern by bit pattern.

The oracle builds its maps by looping over decades and bins (``oracle.qmap``).
Here every 8-bit (and 4-bit) pattern is decoded on its own, the way the
dynamic tree data type of Dettmers et al., "8-bit Optimizers via Block-wise
Quantization" (arXiv:2110.02861) lays a code out: a sign bit (signed maps
only), then E zero bits that set the decade 10^-E, a one bit that ends them,
and the remaining F bits as the index of a linear bin of [0.1, 1] whose centre
is the value.  The two patterns with no terminating one bit carry the two
values the reading adds, 0 and +1.0.  The decoded set must be the oracle's map
value for value: a wrong bit budget (F off by one), a bin edge taken for its
centre, a lost sign or a missing decade would each change it.  (The pages
print no map; this pins the oracle's construction against the published
layout, not the values against the pages.)
"""

from fractions import Fraction

import numpy as np
import pytest

from oracle import qmap

F32 = np.float32


def _round_f32(q: Fraction) -> np.float32:
    """Nearest float32 of an exact rational (ties to even), by exact comparison."""
    c = F32(float(q))
    best = None
    for cand in (np.nextafter(c, F32(-np.inf)), c, np.nextafter(c, F32(np.inf))):
        key = (abs(Fraction(float(cand)) - q), int(np.asarray(cand).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, cand)
    return F32(best[1])


def _decode(pattern: int, bits: int, signed: bool):
    """The value of one code pattern, or the special code it stands for."""
    sign = 1
    body_bits = bits
    if signed:
        sign = -1 if (pattern >> (bits - 1)) & 1 else 1
        body_bits = bits - 1
    body = pattern & ((1 << body_bits) - 1)
    # count the leading zeros of the body
    e = 0
    while e < body_bits and not (body >> (body_bits - 1 - e)) & 1:
        e += 1
    f = body_bits - 1 - e                        # bits after the terminating one
    if f < 0:                                    # no terminating one: a special code
        return ("special", sign)
    k = body & ((1 << f) - 1)
    centre = Fraction(1, 10) + Fraction(2 * k + 1, 2 ** (f + 1)) * Fraction(9, 10)
    return ("value", sign * centre / 10 ** e)


def _decoded_map(bits: int, signed: bool, max_decade: int):
    vals, specials = [], []
    for pat in range(1 << bits):
        kind, x = _decode(pat, bits, signed)
        if kind == "special":
            specials.append(x)
            continue
        e = 0
        while abs(x) * 10 ** (e + 1) <= 1:       # decade of the value
            e += 1
        if e <= max_decade:
            vals.append(_round_f32(x))
        else:
            specials.append(None)                # a decade the map does not use
    return vals, specials


@pytest.mark.parametrize("bits,signed,max_decade,table", [
    (8, True, 6, qmap.signed_map),
    (8, False, 6, qmap.unsigned_map),
    (4, True, 2, qmap.signed_map4),
])
def test_decoded_patterns_are_the_oracle_map(bits, signed, max_decade, table):
    vals, specials = _decoded_map(bits, signed, max_decade)
    # the patterns left over (no terminating one bit, or a decade past the last)
    # hold exactly the two added values
    assert len(vals) + len(specials) == 1 << bits
    assert len(specials) == 2
    full = np.sort(np.array(vals + [F32(0.0), F32(1.0)], dtype=F32))
    assert np.array_equal(full.view(np.uint32), table().view(np.uint32))


def test_decades_and_bin_counts():
    """Per decade of the 8-bit signed map, 2^(6-E) values per sign, spaced 0.9/2^(6-E)
    times 10^-E apart (the linear bins of the layout)."""
    m = qmap.signed_map().astype(np.float64)
    pos = m[m > 0][:-1]                          # +1.0 is the added value
    for e in range(7):
        d = pos[(pos >= 10.0 ** -(e + 1)) & (pos < 10.0 ** -e)]
        assert d.size == 2 ** (6 - e), e
        if d.size > 1:
            # float32 values: each difference within two ulps of the decade's largest value
            assert np.allclose(np.diff(d), 0.9 * 10.0 ** -e / 2 ** (6 - e), rtol=0,
                               atol=2 * 2.0 ** -23 * 10.0 ** -e)
