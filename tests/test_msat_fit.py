"""The M_sat re-fit rule on hand-made timing tables (no GPU): the grid threshold whose dispatch
(dense at M_eff >= M_sat) loses the least time against the faster backend of each cell ("3
GraniKV" per-step dispatch; "Limitations": the threshold is hardware-specific)."""

from shared_prefix_kv_decode_gb300.msat_fit import fit_msat


def _rows(win, slow=2.0):
    rows = []
    for L_p in (512, 2048, 8192):
        for B in (1, 8, 32, 128, 256):
            d, c = (1.0, slow) if win(L_p, B) else (slow, 1.0)
            rows.append({"L_p": L_p, "B": B, "dense_us": d, "cascade_us": c})
    return rows


def test_crossover_at_first_winning_meff():
    assert fit_msat(_rows(lambda L, B: B >= 32)) == 128


def test_majority_of_cells_decides():
    # dense loses at L_p = 512 for every B but wins above 2048 from B = 8 on: the threshold
    # B = 8 (M_eff 32) gives up four short-prefix cells and keeps eight long-prefix ones
    assert fit_msat(_rows(lambda L, B: L >= 2048 and B >= 8)) == 32


def test_one_loss_above_does_not_move_the_threshold():
    # dense wins from B = 32 on except one cell (B = 128, L_p = 8192)
    assert fit_msat(_rows(lambda L, B: (B >= 32 and not (B == 128 and L == 8192)))) == 128


def test_many_losses_above_move_it():
    # dense loses at B = 32 and 128 for every L_p, wins only at B = 256
    assert fit_msat(_rows(lambda L, B: B >= 256 or B == 8)) == 1024


def test_always_and_never():
    assert fit_msat(_rows(lambda L, B: True)) == 4
    assert fit_msat(_rows(lambda L, B: False)) > 4 * 256


def test_committed_gb300_sweep_fits_the_built_in_threshold():
    """The GB300 sweep committed with the package (the table the built-in M_sat comes from): the
    least-regret fit gives the library's default M_sat of 4 (the dense backend from the smallest
    M_eff of the grid), the recorded strict-rule threshold is what the strict rule gives on the
    table, and the dispatched call is within 2 % of the faster single backend in every cell
    ("3 GraniKV", per-step dispatch: never slower than either backend alone)."""
    import json
    import os
    from shared_prefix_kv_decode_gb300 import msat_fit as MF
    path = os.path.join(os.path.dirname(MF.__file__), "msat_gb300.json")
    with open(path) as f:
        d = json.load(f)
    rows = d["rows"]
    assert len(rows) == 30 and {r["L_p"] for r in rows} == {512, 2048, 8192, 16384, 32768}
    assert MF.fit_msat(rows) == d["m_sat"] == 4
    assert MF.fit_msat_strict(rows) == d["m_sat_strict"]
    worst = max(rows, key=MF.dispatch_ratio)
    assert MF.dispatch_ratio(worst) <= 1.02, worst


def test_strict_rule_on_hand_tables():
    from shared_prefix_kv_decode_gb300.msat_fit import fit_msat_strict
    # dense wins from B = 32 on at every L_p >= 2048, loses below (the L_p = 512 row is ignored)
    rows = _rows(lambda L, B: B >= 32 or L == 512)
    assert fit_msat_strict(rows) == 128
    # one loss at B = 128 (L_p 8192) pushes the strict threshold past it
    rows = _rows(lambda L, B: B >= 32 and not (B == 128 and L == 8192))
    assert fit_msat_strict(rows) == 1024
