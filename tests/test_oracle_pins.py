"""The CPU oracle against its pins (closed forms, brute force, finite differences, invariants)."""
import pytest

from oracle import vloss_oracle as O
from tests import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    if pin.__name__ in ("pin_ce_brute_force", "pin_ce_mean_page_case", "pin_kl_brute_force",
                        "pin_topk_probs_full_softmax"):
        pytest.importorskip("mpmath")
    pin(O)


def test_memory_figure():
    P.pin_memory_figure()
