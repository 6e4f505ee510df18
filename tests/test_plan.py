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


def _check_invariants(M, N, K, pairs, plan):
    T = plan["tiles_m"] * plan["tiles_n"]
    assert plan["tiles_m"] == -(-M // 256) and plan["tiles_n"] == -(-N // plan["tile_n"])
    assert plan["k_stages"] == -(-K // 32)
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
    fwd = emu.emu_plan_query(6144, 1024, 256, GB300_PAIRS)   # 96 tiles of 8 k-stages
    assert (fwd["tiles_a"], fwd["split_a"], fwd["split_b"], fwd["units"], fwd["pairs"]) == (76, 1, 3, 136, 76)
    assert fwd["pipe"] == 0 and fwd["slots"] == 60
    dx = emu.emu_plan_query(6144, 256, 1024, GB300_PAIRS)    # 24 tiles of 32 k-stages
    assert (dx["tiles_a"], dx["split_a"], dx["units"], dx["pairs"], dx["slots"]) == (24, 3, 72, 72, 72)
    large = emu.emu_plan_query(552960, 1024, 256, GB300_PAIRS)
    assert large["slots"] == 0 and large["units"] == 2160 * 4 and large["pairs"] == GB300_PAIRS


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


def test_plan_query_rejects_bad_arguments():
    for args in [(0, 1, 1, 76), (1, 0, 1, 76), (1, 1, 0, 76), (1, 1, 1, 0), (-5, 1, 1, 76)]:
        with pytest.raises(emu.EmuError) as e:
            emu.emu_plan_query(*args)
        assert e.value.status == 1


def _cost(plan, pairs):
    """Predicted time in pipeline stages, from the plan's own fields: waves
    of units, each its k-stages plus 3 stages of output stores, plus 1.5
    stages of reduction when a tile is split."""
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
    c = _cost(plan, GB300_PAIRS)
    assert abs(plan["cost_x100"] / 100.0 - c) <= 0.006
    T, KS = plan["tiles_m"] * plan["tiles_n"], plan["k_stages"]
    assert c <= -(-T // GB300_PAIRS) * (KS + 3) + 1e-9
