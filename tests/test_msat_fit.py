"""The M_sat re-fit rule on hand-made timing tables (no GPU): the smallest grid M_eff at which
dense is no slower than cascade for every L_p >= 2048, at that M_eff and all larger ones
("3 GraniKV" per-step dispatch; "Limitations": the threshold is hardware-specific)."""

from shared_prefix_kv_decode_gb300.msat_fit import fit_msat


def _rows(win):
    rows = []
    for L_p in (512, 2048, 8192):
        for B in (1, 8, 32, 128, 256):
            d, c = (1.0, 2.0) if win(L_p, B) else (2.0, 1.0)
            rows.append({"L_p": L_p, "B": B, "dense_us": d, "cascade_us": c})
    return rows


def test_crossover_at_first_winning_meff():
    assert fit_msat(_rows(lambda L, B: B >= 32)) == 128


def test_short_prefixes_do_not_count():
    # dense loses at L_p = 512 for every B but wins above 2048 from B = 8 on
    assert fit_msat(_rows(lambda L, B: L >= 2048 and B >= 8)) == 32


def test_a_loss_above_moves_the_threshold_up():
    # dense wins at B = 32 but loses again at B = 128 (one L_p), so only B >= 256 qualifies
    assert fit_msat(_rows(lambda L, B: (B >= 32 and not (B == 128 and L == 8192)))) == 1024


def test_never_wins():
    assert fit_msat(_rows(lambda L, B: False)) is None
