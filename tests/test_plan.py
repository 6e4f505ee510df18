"""The launch planner (host logic, no GPU): how tiles become work units.

A split tile's pieces wait for one another on the GPU, so every plan must
put all pieces of a split tile in the same wave of units; the counts the
kernel relies on (units, pairs, workspace partial tiles) must add up.
"""
import itertools

import pytest

import fp32_emulated_gemm_gb300 as emu

GB300_PAIRS = 76


def _units(plan):
    """(tile, piece, pieces) of every work unit, in unit order."""
    T = plan["tiles_m"] * plan["tiles_n"]
    out = []
    for t in range(plan["tiles_a"]):
        out += [(t, q, plan["split_a"]) for q in range(plan["split_a"])]
    for t in range(plan["tiles_a"], T):
        out += [(t, q, plan["split_b"]) for q in range(plan["split_b"])]
    return out


def _chain_runs(plan, bounds):
    """Chained plans, as the header states them: pair c runs the stages
    [b_c, b_c+1) of the U = T KS stages taken tile by tile, each tile's in
    decreasing k order.  Per pair, its units in order as (tile, kb, ke): the
    k-stages [kb, ke) of the tile, run in increasing k."""
    KS = plan["k_stages"]
    runs = []
    for c in range(plan["pairs"]):
        s, e = bounds[c], bounds[c + 1]
        units = []
        for t in range(s // KS, (e - 1) // KS + 1):
            lo, hi = max(s, t * KS) - t * KS, min(e, (t + 1) * KS) - t * KS
            units.append((t, KS - hi, KS - lo))
        runs.append(units)
    return runs


def _run_cost(units, KS):
    """The planner's cost of one pair's run, in pipeline stages: its stages,
    plus a cost for each step from one unit to the next by the kinds of the
    two units (head = the low k-stages of a cut tile, tail = its high ones,
    whole = an uncut tile): head -> whole 1.1, head -> tail 1.6,
    whole -> whole 2, whole -> tail 4."""
    def kind(kb, ke):
        return "head" if kb == 0 and ke < KS else ("tail" if ke == KS and kb > 0 else "whole")
    step = {("head", "whole"): 1.1, ("head", "tail"): 1.6, ("whole", "whole"): 2.0, ("whole", "tail"): 4.0}
    kinds = [kind(kb, ke) for (_, kb, ke) in units]
    return sum(ke - kb for (_, kb, ke) in units) + sum(step[(a, b)] for a, b in zip(kinds, kinds[1:]))


def _check_chain(M, N, K, pairs, plan):
    import fp32_emulated_gemm_gb300 as emu
    T, KS, P = plan["tiles_m"] * plan["tiles_n"], plan["k_stages"], plan["pairs"]
    assert P == pairs and T >= P
    assert (plan["tiles_a"], plan["split_a"], plan["split_b"]) == (T, 1, 1)
    bounds = emu.emu_plan_bounds(M, N, K, pairs)
    U = T * KS
    assert bounds[0] == 0 and bounds[-1] == U and len(bounds) == P + 1
    for c in range(1, P):                                             # near the even cut, increasing
        assert abs(bounds[c] - c * U // P) <= 2 and bounds[c] > bounds[c - 1]
    runs = _chain_runs(plan, bounds)
    covered = {}
    for c, r in enumerate(runs):
        assert r, f"pair {c} has no work"
        for i, (t, kb, ke) in enumerate(r):
            assert 0 <= kb < ke <= KS
            for k in range(kb, ke):
                assert (t, k) not in covered
                covered[(t, k)] = (c, i)
    assert len(covered) == T * KS                                     # every stage of every tile, once
    cuts = 0
    for t in range(T):
        owners = sorted({covered[(t, k)][0] for k in range(KS)})
        assert len(owners) in (1, 2)                                  # no tile cut twice
        if len(owners) == 2:
            cuts += 1
            c = owners[0]
            assert owners[1] == c + 1
            # the next pair runs the low k-stages as its first unit (it waits
            # for nothing); this pair runs the high ones as its last unit,
            # after all its other work, from the published running sum
            assert runs[c + 1][0][0] == t and runs[c + 1][0][1] == 0
            assert runs[c][-1][0] == t and runs[c][-1][2] == KS
            assert runs[c][-1][1] == runs[c + 1][0][2]
    assert plan["units"] == sum(len(r) for r in runs)
    assert plan["slots"] == (P - 1 if cuts else 0)
    cost = max(_run_cost(r, KS) for r in runs)
    assert abs(plan["cost_x100"] / 100.0 - cost) <= 0.006
    # no worse than the even cuts, where those are valid
    even = [c * U // P for c in range(P + 1)]
    even_runs = _chain_runs(plan, even)
    if all(len(r) > 1 or r[0][1] == 0 or r[0][2] == KS for r in even_runs):
        assert cost <= max(_run_cost(r, KS) for r in even_runs) + 1e-9


def _check_invariants(M, N, K, pairs, plan):
    T = plan["tiles_m"] * plan["tiles_n"]
    assert plan["tiles_m"] == -(-M // 256) and plan["tiles_n"] == -(-N // plan["tile_n"])
    assert plan["k_stages"] == -(-K // 32)
    if plan["chain"]:
        _check_chain(M, N, K, pairs, plan)
        return
    units = _units(plan)
    assert plan["units"] == len(units)
    assert 1 <= plan["pairs"] <= min(pairs, plan["units"])
    for S in (plan["split_a"], plan["split_b"]):
        assert 1 <= S <= min(32, plan["k_stages"], pairs)
    slots = sum(1 for (_, _, S) in units if S > 1)
    assert plan["slots"] == slots
    # pieces of one split tile: consecutive units in one wave, each >= 1 k-stage
    by_tile = {}
    for u, (t, q, S) in enumerate(units):
        by_tile.setdefault(t, []).append((u, q, S))
    assert sorted(by_tile) == list(range(T))
    for t, us in by_tile.items():
        S = us[0][2]
        assert [q for (_, q, _) in us] == list(range(S))
        waves = {u // plan["pairs"] for (u, _, _) in us}
        assert len(waves) == 1, f"tile {t} straddles waves"
        for (_, q, _) in us:
            kb = q * plan["k_stages"] // S
            ke = (q + 1) * plan["k_stages"] // S
            assert ke > kb


SHAPES = [(6144, 1024, 256), (6144, 256, 1024), (552960, 1024, 256), (552960, 256, 1024),
          (6144, 4096, 1024), (6144, 1024, 4096), (128, 128, 256), (256, 256, 256), (1024, 1024, 1024),
          (4096, 4096, 4096), (16384, 16384, 16384), (1, 1, 1), (300, 260, 3000), (2048, 2048, 65536),
          (257, 1, 64), (38912, 1024, 4096)]


@pytest.mark.parametrize("pairs", [GB300_PAIRS, 74, 37, 5, 1])
def test_plans_keep_split_tiles_in_one_wave(pairs):
    for (M, N, K) in SHAPES:
        _check_invariants(M, N, K, pairs, emu.emu_plan_query(M, N, K, pairs))


def test_pet_plans():
    # forward: 96 tiles of 8 k-stages, chained: runs of 10-11 stages on all
    # 76 pairs (whole tiles and a 3-way split tail would take 8 + 3 stages
    # and a reduce-scatter)
    fwd = emu.emu_plan_query(6144, 1024, 256, GB300_PAIRS)
    assert (fwd["chain"], fwd["tiles_a"], fwd["split_a"], fwd["split_b"], fwd["pairs"]) == (1, 96, 1, 1, 76)
    assert fwd["pipe"] == 0 and fwd["slots"] == GB300_PAIRS - 1
    _check_invariants(6144, 1024, 256, GB300_PAIRS, fwd)
    # input gradient: 24 tiles of 32 k-stages, fewer than the pairs: 3 pieces each
    dx = emu.emu_plan_query(6144, 256, 1024, GB300_PAIRS)
    assert (dx["chain"], dx["tiles_a"], dx["split_a"], dx["units"], dx["pairs"], dx["slots"]) == (0, 24, 3, 72, 72, 72)
    # PET-large: 8640 tiles, 113.7 per pair: chained
    large = emu.emu_plan_query(552960, 1024, 256, GB300_PAIRS)
    assert large["chain"] == 1 and large["pairs"] == GB300_PAIRS and large["slots"] == GB300_PAIRS - 1
    _check_invariants(552960, 1024, 256, GB300_PAIRS, large)
    # the wide layers' 96-tile products: 161-162 stages per pair instead of
    # 128 + 43 for whole tiles and a 3-way tail
    wide = emu.emu_plan_query(6144, 1024, 4096, GB300_PAIRS)
    assert wide["chain"] == 1 and wide["slots"] == GB300_PAIRS - 1
    # a whole number of waves: no tile would be cut, round-robin whole tiles
    even = emu.emu_plan_query(38912, 1024, 4096, GB300_PAIRS)
    assert (even["chain"], even["slots"], even["units"]) == (0, 0, 608)


def test_overrides(monkeypatch):
    monkeypatch.setenv("EMU_SPLIT_K", "5")
    p = emu.emu_plan_query(6144, 1024, 4096, GB300_PAIRS)
    assert (p["tiles_a"], p["split_a"]) == (96, 5)
    _check_invariants(6144, 1024, 4096, GB300_PAIRS, p)
    monkeypatch.setenv("EMU_SPLIT_K", "100")        # capped at 32 pieces
    assert emu.emu_plan_query(6144, 1024, 4096, GB300_PAIRS)["split_a"] == 32
    monkeypatch.delenv("EMU_SPLIT_K")
    monkeypatch.setenv("EMU_PIPE", "1")
    assert emu.emu_plan_query(6144, 1024, 256, GB300_PAIRS)["pipe"] == 1
    monkeypatch.delenv("EMU_PIPE")
    auto = emu.emu_plan_query(6144, 1024, 256, GB300_PAIRS)
    monkeypatch.setenv("EMU_SPLIT_TAIL", "2")       # hybrid tail in 2 pieces
    p = emu.emu_plan_query(6144, 1024, 256, GB300_PAIRS)
    assert (p["tiles_a"], p["split_a"], p["split_b"], p["units"]) == (76, 1, 2, 116)
    _check_invariants(6144, 1024, 256, GB300_PAIRS, p)
    monkeypatch.setenv("EMU_SPLIT_TAIL", "4")       # 20 tail tiles x 4 > 76 pairs: not a valid wave, ignored
    assert emu.emu_plan_query(6144, 1024, 256, GB300_PAIRS) == auto
    monkeypatch.delenv("EMU_SPLIT_TAIL")
    dx = emu.emu_plan_query(6144, 256, 1024, GB300_PAIRS)
    monkeypatch.setenv("EMU_SPLIT_TAIL", "2")       # 24 tiles < 76 pairs: no hybrid plan exists, ignored
    assert emu.emu_plan_query(6144, 256, 1024, GB300_PAIRS) == dx
    monkeypatch.delenv("EMU_SPLIT_TAIL")
    monkeypatch.setenv("EMU_CHAIN", "1")            # chained wherever tiles >= pairs
    fwd = emu.emu_plan_query(6144, 1024, 256, GB300_PAIRS)
    assert fwd["chain"] == 1 and fwd["units"] > 96 and fwd["slots"] == GB300_PAIRS - 1
    _check_invariants(6144, 1024, 256, GB300_PAIRS, fwd)
    assert emu.emu_plan_query(6144, 256, 1024, GB300_PAIRS) == dx      # 24 tiles: not possible, ignored
    monkeypatch.setenv("EMU_SPLIT_K", "2")          # an explicit split wins
    assert emu.emu_plan_query(6144, 1024, 256, GB300_PAIRS)["chain"] == 0
    monkeypatch.delenv("EMU_SPLIT_K")
    monkeypatch.setenv("EMU_CHAIN", "2")            # chained, the even cuts c U / P
    even = emu.emu_plan_query(6144, 1024, 256, GB300_PAIRS)
    assert even["chain"] == 1
    assert emu.emu_plan_bounds(6144, 1024, 256, GB300_PAIRS) == [c * 768 // 76 for c in range(77)]
    _check_invariants(6144, 1024, 256, GB300_PAIRS, even)
    monkeypatch.setenv("EMU_CHAIN", "0")            # never chained
    assert emu.emu_plan_query(6144, 1024, 4096, GB300_PAIRS)["chain"] == 0
    with pytest.raises(emu.EmuError) as e:          # bounds exist only for chained plans
        emu.emu_plan_bounds(6144, 1024, 4096, GB300_PAIRS)
    assert e.value.status == 2


def test_plan_query_rejects_bad_arguments():
    for args in [(0, 1, 1, 76), (1, 0, 1, 76), (1, 1, 0, 76), (1, 1, 1, 0), (-5, 1, 1, 76)]:
        with pytest.raises(emu.EmuError) as e:
            emu.emu_plan_query(*args)
        assert e.value.status == 1


def _cost(plan, pairs):
    """Predicted time in pipeline stages, from the plan's own fields: waves
    of units, each its k-stages plus 3 stages of output stores, plus 1.5
    stages of reduction when a tile is split (chained plans: see
    _check_chain)."""
    T, KS = plan["tiles_m"] * plan["tiles_n"], plan["k_stages"]
    Sa, Sb = plan["split_a"], plan["split_b"]
    if Sb == 1 and plan["tiles_a"] == T:
        units = T * Sa
        used = pairs if (units <= pairs or Sa == 1) else pairs // Sa * Sa
        return -(-units // used) * (-(-KS // Sa) + 3) + (1.5 if Sa > 1 else 0.0)
    W = plan["tiles_a"] // pairs
    return W * (KS + 3) + (-(-KS // Sb) + 3) + 1.5


@pytest.mark.parametrize("M,N,K", [(6144, 1024, 256), (6144, 256, 1024), (552960, 1024, 256), (64, 64, 64),
                                   (1536, 256, 1024), (2048, 2048, 2048), (19 * 256, 4 * 256, 4096)])
def test_plan_cost_is_reported_and_no_worse_than_unsplit(M, N, K):
    plan = emu.emu_plan_query(M, N, K, GB300_PAIRS)
    if plan["chain"]:
        _check_invariants(M, N, K, GB300_PAIRS, plan)
        return
    c = _cost(plan, GB300_PAIRS)
    assert abs(plan["cost_x100"] / 100.0 - c) <= 0.006
    T, KS = plan["tiles_m"] * plan["tiles_n"], plan["k_stages"]
    assert c <= -(-T // GB300_PAIRS) * (KS + 3) + 1e-9
