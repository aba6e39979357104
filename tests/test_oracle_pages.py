"""Pin of the page-movement ordering model against the Fig. 4 walk-through (CPU only)."""
import pytest

from conftest import load_golden
from oracle import pages


def _apply(bp, op, arg):
    if op == "offload":
        return bp.offload(arg)
    if op == "reload":
        return bp.reload(arg)
    if op == "landed":
        return bp.copies_landed()
    if op == "commit":
        return bp.commit()
    if op == "set_bits":
        return bp.set_bits(arg)
    raise ValueError(op)


def test_fig4_walkthrough():
    g = load_golden("fig4_scenario.json")
    bp = pages.BlockPages(g["bits"], g["bmax"], g["q0"])
    for ev in g["events"]:
        r = _apply(bp, ev["op"], ev.get("arg"))
        if "applied" in ev:
            assert r == ev["applied"]
        assert bp.q == ev["q"], ev
        assert bp.state == ev["state"], ev


def test_illegal_orders():
    g = load_golden("fig4_scenario.json")
    for case in g["illegal"]:
        bp = pages.BlockPages(g["bits"], g["bmax"], case["q0"])
        for n, (op, arg) in enumerate(case["ops"]):
            if n == case["error_at"]:
                with pytest.raises(pages.StateError):
                    _apply(bp, op, arg)
                break
            _apply(bp, op, arg)


def test_offload_lowers_before_move_and_reload_raises_after():
    bp = pages.BlockPages((3, 4, 5, 6, 7, 8), 8, 8)
    bp.offload(5)
    assert bp.q == 5 and bp.state[5:] == ["to_cpu"] * 3
    bp.copies_landed()
    bp.reload(8)
    assert bp.q == 5  # not raised while in transfer
    assert bp.commit() == 0
    bp.copies_landed()
    assert bp.commit() == 1 and bp.q == 8
