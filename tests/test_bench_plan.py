"""The benchmark's replay plan: the timed region runs exactly the requested
number of steps, whole round graphs first, and the cache copies follow each
other round-robin (so every copy is touched as often as the others, give or
take one, and the L2 never holds the copy about to be read)."""
import bench


def _steps(plan, R):
    """Expand a plan into the cache copy of every step."""
    out = []
    for g in plan:
        if g == "round":
            out += [i % R for i in range(bench.round_steps(R))]
        else:
            out.append(g)
    return out


def test_round_steps_are_whole_passes_near_16():
    for R in range(1, 40):
        rs = bench.round_steps(R)
        assert rs % R == 0 and rs >= R
        assert rs <= max(16, R)


def test_plan_counts_exactly_the_steps():
    for R in (1, 2, 3, 4, 5, 7, 16, 20):
        for n in (0, 1, 3, 15, 16, 17, 20, 50, 101):
            for use_round in (True, False):
                plan = bench.replay_plan(n, R, use_round)
                copies = _steps(plan, R)
                assert len(copies) == n, (R, n, use_round)
                assert all(0 <= c < R for c in copies)
                if not use_round:
                    assert "round" not in plan


def test_plan_rounds_first_then_round_robin_copies():
    R, n = 4, 50
    plan = bench.replay_plan(n, R)
    rounds = plan.count("round")
    assert plan[:rounds] == ["round"] * rounds and "round" not in plan[rounds:]
    assert rounds == n // bench.round_steps(R)
    copies = _steps(plan, R)
    # each step's copy differs from the previous one's (R > 1), and the
    # copies are used evenly
    assert all(a != b for a, b in zip(copies, copies[1:]))
    counts = [copies.count(r) for r in range(R)]
    assert max(counts) - min(counts) <= 1
