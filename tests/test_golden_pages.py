"""Pin the communication-volume arithmetic to the figures the pages print
(fixture: tests/golden/pages_byte_counts.txt, each line cited there)."""
import os
from decimal import Decimal

import pytest

from oracle import comm_volume as C

HERE = os.path.dirname(os.path.abspath(__file__))


def _rows():
    with open(os.path.join(HERE, "golden", "pages_byte_counts.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kind, tokens, V, t, elem, printed, unit, src = line.split()
            yield kind, int(tokens), int(V), int(t), int(elem), printed, unit, src


UNIT = {"GB": Decimal(10) ** 9, "MB": Decimal(10) ** 6, "x": Decimal(1), "cols": Decimal(1)}


def _matches_printed(value, printed):
    """The page prints a figure to a few digits, rounded or cut off."""
    from decimal import ROUND_DOWN, ROUND_HALF_UP
    q = Decimal(1).scaleb(Decimal(printed).as_tuple().exponent)
    v = Decimal(value)
    return Decimal(printed) in (v.quantize(q, rounding=ROUND_HALF_UP), v.quantize(q, rounding=ROUND_DOWN))


@pytest.mark.parametrize("row", list(_rows()), ids=lambda r: f"{r[0]}-{r[2]}-{r[7]}")
def test_printed_byte_counts(row):
    kind, tokens, V, t, elem, printed, unit, _ = row
    if kind == "allgather_logits":
        val = Decimal(C.allgather_logits_bytes(tokens, V, t, elem).numerator) / \
            Decimal(C.allgather_logits_bytes(tokens, V, t, elem).denominator)
    elif kind == "fused_ce":
        f = C.fused_ce_bytes(tokens, t, 3, elem)
        val = Decimal(f.numerator) / Decimal(f.denominator)
    elif kind in ("ratio", "ratio_approx"):
        r = C.allgather_logits_bytes(tokens, V, t, elem) / C.fused_ce_bytes(tokens, t)
        val = Decimal(r.numerator) / Decimal(r.denominator)
    elif kind == "logits":
        val = Decimal(C.logits_bytes(tokens, V, elem))
    elif kind == "columns_per_card":
        val = Decimal(C.columns_per_card(V, t))
    else:
        raise AssertionError(kind)
    scaled = val / UNIT[unit]
    if kind == "ratio_approx":  # printed as "about 5300": two significant digits
        assert round(scaled, -2) == Decimal(printed)
    else:
        assert _matches_printed(scaled, printed), (scaled, printed)


def test_indivisible_vocab_needs_padding():
    # "LLM Internals" §7.3.7: a vocabulary not divisible by t cannot be split evenly
    with pytest.raises(ValueError):
        C.columns_per_card(50257, 8)
